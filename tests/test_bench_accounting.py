"""The benchmark's algorithmic work counts (host logic, no GPU): FLOPs per visible (query, key)
pair and bytes per decode call, checked against brute-force counts on small shapes and pinned at
the benchmarked shapes."""
import itertools

import pytest

import bench
import synth_inputs as si


def _visible_pairs(nq, nk, causal):
    return sum(1 for i, j in itertools.product(range(nq), range(nk)) if not causal or j <= i)


@pytest.mark.parametrize("n", [1, 2, 5, 17])
def test_causal_counts_match_brute_force(n):
    b, h, d = 2, 3, 8
    pairs = _visible_pairs(n, n, True)
    assert bench.causal_attn_flops(b, h, n, d) == pytest.approx(4 * d * b * h * pairs)
    assert bench.causal_attn_bwd_flops(b, h, n, d) == pytest.approx(10 * d * b * h * pairs)
    assert bench.dense_attn_flops(b, h, n, n + 3, d) == pytest.approx(4 * d * b * h * _visible_pairs(n, n + 3, False))


def test_varlen_flops_sum_per_sequence():
    lens, h, d = [3, 1, 4], 2, 8
    pairs = sum(_visible_pairs(n, n, True) for n in lens)
    assert bench.varlen_causal_flops(lens, h, d) == pytest.approx(4 * d * h * pairs)


def test_decode_bytes_count_every_tensor_once():
    b, h, d, kv = 1, 2, 4, [5]
    # bf16 q and o (b h d each), K and V rows of the visible keys, fp32 LSE per (b, h)
    mha = 2 * (b * h * d) * 2 + 2 * (2 * h * d * sum(kv)) + 4 * b * h
    assert bench.decode_bytes(b, h, d, sum(kv)) == mha
    gqa = 2 * (b * h * d) * 2 + 2 * (2 * 1 * d * sum(kv)) + 4 * b * h  # one key/value head
    assert bench.decode_bytes(b, h, d, sum(kv), h_kv=1) == gqa


def test_benchmarked_workloads():
    # the figures the benchmark reports as algorithmic work
    assert bench.causal_attn_bwd_flops(1, 32, 8192, 128) == pytest.approx(1374557306880.0)
    kv = int(si.decode_kv_len(32, 32768, seed=0).sum())
    assert bench.decode_bytes(32, 32, 128, kv) == pytest.approx(16241020928.0)
    assert bench.decode_bytes(32, 32, 128, kv, h_kv=8) == pytest.approx(4060651520.0)
    lens = si.varlen_lengths(16, 8192, seed=0, min_len=1024)
    assert bench.varlen_causal_flops(lens, 32, 128) == pytest.approx(5170632589312.0)


@pytest.mark.parametrize("nq,nk", [(1, 1), (1, 9), (3, 7), (5, 5), (17, 40), (7, 3)])
def test_kvcache_causal_counts_match_brute_force(nq, nk):
    # the queries are the last nq positions of nk keys: query i sees keys j <= i + (nk - nq)
    pairs = sum(1 for i, j in itertools.product(range(nq), range(nk)) if j <= i + nk - nq)
    assert bench.causal_pairs(nq, nk) == pairs
    assert bench.kvcache_causal_flops(2, 3, nq, nk, 8) == pytest.approx(4 * 8 * 2 * 3 * pairs)
    if nq == nk:
        assert bench.kvcache_causal_flops(2, 3, nq, nk, 8) == pytest.approx(bench.causal_attn_flops(2, 3, nq, 8))


def test_dense_bwd_flops():
    assert bench.dense_attn_bwd_flops(4, 16, 4096, 4096, 64) == pytest.approx(2.5 * 4 * 4 * 16 * 4096 * 4096 * 64)


def test_time_floor_repeats():
    # the K-step loop repeats until the timed region reaches the floor
    assert bench.repeats_for(3.0, 20, 0.38) == 395  # ceil(3000 / 7.6)
    assert bench.repeats_for(3.0, 400, 10.0) == 1
    assert bench.repeats_for(0.0, 20, 0.38) == 1
    r = bench.repeats_for(2.0, 20, 0.38)
    assert r * 20 * 0.38 >= 2000.0 and (r - 1) * 20 * 0.38 < 2000.0


def test_clock_line_parsing():
    line = "0, 1965, 2070, 1012.55, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
    sm, smax, pw, act = bench.ClockSampler.parse(line)
    assert (sm, smax, pw) == (1965.0, 2070.0, 1012.55)
    assert act == {"hw_slowdown": False, "hw_thermal_slowdown": False, "sw_thermal_slowdown": False,
                   "sw_power_cap": True}
    assert bench.ClockSampler.parse("0, [N/A], 2070, 5, x, a, b, c, d") is None
    assert bench.ClockSampler.parse("garbage") is None


def test_both_arms_report_the_same_config():
    import inspect
    src = inspect.getsource(bench.main_reference) + inspect.getsource(bench.main)
    assert src.count("headline_config(world)") == 2
    cfg = bench.headline_config(1)
    assert cfg["Nq"] == cfg["Nk"] == 8192 and cfg["causal"] is True and "parallelism" in cfg


def test_case_table_covers_the_components():
    assert set(bench.COMPONENTS) | {"attn_causal"} == set(bench.CASES)
    assert "attn_bwd_noncausal_d64" in bench.COMPONENTS and "attn_decode_gqa" in bench.COMPONENTS


def test_chunked_prefill_work():
    # 2048 queries at the end of 32768 keys: query i sees 30721 + i keys
    pairs = sum(30721 + i for i in range(2048))
    assert bench.causal_pairs(2048, 32768) == pairs == 65012736
    assert bench.kvcache_causal_flops(8, 32, 2048, 32768, 128) == pytest.approx(4 * 128 * 8 * 32 * pairs)


def test_multi_token_decode_bytes():
    b, h, d, kv, nq = 2, 4, 8, [5, 3], 3
    # bf16 q and o (b h nq d each), K and V of the visible keys over one key/value head, fp32 LSE per row
    want = 2 * (b * h * nq * d) * 2 + 2 * (2 * 1 * d * sum(kv)) + 4 * b * h * nq
    assert bench.decode_bytes(b, h, d, sum(kv), h_kv=1, nq=nq) == want
    assert bench.decode_bytes(b, h, d, sum(kv), h_kv=1) == bench.decode_bytes(b, h, d, sum(kv), h_kv=1, nq=1)


def test_code_digest_ignores_comments_but_not_code():
    src = "int a = 1;  // the first\n\n// a note\nint b = a + 2;\n"
    same = "int a = 1;   // reworded\n// another note\n\n\nint b = a + 2;\n"
    changed = "int a = 1;\nint b = a + 3;\n"
    assert bench.code_digest([src]) == bench.code_digest([same])
    assert bench.code_digest([src]) != bench.code_digest([changed])
    # the files' order and boundaries count
    assert bench.code_digest(["int a = 1;", "int b;"]) != bench.code_digest(["int b;", "int a = 1;"])


def test_profiled_traffic_needs_the_current_digest(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = tmp_path / "online_softmax_attention_tiled_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "attn_tc.cu").write_text("int k = 1;  // kernel\n")
    (csrc / "oa_common.cuh").write_text("int c = 2;\n")
    dig = bench.kernel_source_digest()
    f = prof / "attn_fwd_tc_causal_b1h32n8192d128.md"
    f.write_text(f"kernel_source_digest: {dig}\ndram_bytes_per_launch: 1234\n")
    assert bench.profiled_traffic() == 1234.0
    (csrc / "attn_tc.cu").write_text("int k = 1;  // kernel, comment reworded\n")
    assert bench.profiled_traffic() == 1234.0
    (csrc / "attn_tc.cu").write_text("int k = 2;\n")
    assert bench.profiled_traffic() is None
