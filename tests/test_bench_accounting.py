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
