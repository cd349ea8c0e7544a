"""Causal attention of Nq new queries against Nk keys (chunked prefill, multi-token decode against a
KV cache) vs the fp64 oracle (gpu).

The queries are the last Nq positions of the Nk keys' sequence, so query i sees keys
j <= i + (Nk - Nq) (bottom-right alignment; for packed sequences with each sequence's own
lengths).  With Nq > Nk the first Nq - Nk queries see nothing: O = +0.0, LSE = -inf.
Covers the tensor-core forward (both query-tile slots per item, and the split-slot instance for
at most 128 query rows), grouped key/value heads, packed sequences, the fp32 forward and the
benchmarked chunked-prefill shape at sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import BF16_O_ATOL, F32_ATTN_ATOL, assert_lse_close, assert_out_close, bf16_bits

pytestmark = pytest.mark.gpu


def _sync(oa):
    torch.cuda.synchronize()
    oa.sync_status()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq", [1, 17, 128, 300, 2048])
def test_dense_queries_at_the_end_of_an_8192_key_cache(cuda_lib, d, Nq):
    B, H, Nk = 2, 2, 8192
    q, k, v = si.attn_inputs(B, H, Nq, Nk, d, torch.bfloat16, seed=100 + Nq + d)
    kv_len = [Nk, 5000]  # the second sequence's cache is shorter than the tensor: its tail is hidden
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True,
                               kv_len=torch.tensor(kv_len, dtype=torch.int32).cuda())
    _sync(cuda_lib)
    if Nq <= 300:
        ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True, kv_len=kv_len)
        assert_lse_close(lse, rl)
        assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)
    else:  # sampled rows: both sides of every tile boundary and seeded fill, every (b, h)
        rows_i = si.sample_rows(Nq, 160, seed=Nq).numpy()
        flat = np.concatenate([(bh * Nq) + rows_i for bh in range(B * H)])
        ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True, kv_len=kv_len, rows=flat)
        assert_lse_close(lse.reshape(-1)[torch.from_numpy(flat).cuda()], rl)
        assert_out_close(o.reshape(-1, d)[torch.from_numpy(flat).cuda()], ro, BF16_O_ATOL, lse_ref=rl)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(300, 100), (257, 129), (5, 3), (130, 1)])
def test_dense_more_queries_than_keys(cuda_lib, d, Nq, Nk):
    # the first Nq - Nk queries see no key at all
    q, k, v = si.attn_inputs(1, 3, Nq, Nk, d, torch.bfloat16, seed=7 * Nq + Nk + d)
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    _sync(cuda_lib)
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True)
    assert np.isneginf(rl[:, :, :Nq - Nk]).all()
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(4, 1000), (300, 1000), (129, 777)])
def test_grouped_heads_against_a_cache(cuda_lib, d, Nq, Nk):
    B, H, Hkv = 2, 8, 2
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, Nq, Nk, d, torch.bfloat16, seed=200 + Nq + d)
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    _sync(cuda_lib)
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True)
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)


def test_one_query_causal_is_the_whole_cache(cuda_lib):
    # one new query is the last position: causal and non-causal attention are the same call
    q, k, v = si.attn_inputs_gqa(3, 8, 2, 1, 900, 128, torch.bfloat16, seed=301)
    kv = torch.tensor([900, 1, 333], dtype=torch.int32).cuda()
    oc, lc = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, kv_len=kv)
    on, ln_ = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=False, kv_len=kv)
    _sync(cuda_lib)
    assert torch.equal(oc, on) and torch.equal(lc, ln_)


@pytest.mark.parametrize("d", [64, 128])
def test_packed_sequences_against_their_caches(cuda_lib, d):
    # per sequence: more keys than queries (a chunk after its cache), equal, fewer (leading queries see
    # nothing), one query, a sequence without queries and one without keys
    lq = [100, 300, 1, 0, 257, 500, 64, 40]
    lk = [1000, 300, 77, 50, 129, 400, 2000, 0]
    q, k, v, cq, ck = si.varlen_inputs(lq, lk, 4, 2, d, torch.bfloat16, seed=400 + d)
    o, lse = cuda_lib.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), max(lq), max(lk),
                                      causal=True)
    _sync(cuda_lib)
    ro, rl = oracle.attention_varlen(bf16_bits(q), bf16_bits(k), bf16_bits(v), cq.numpy(), ck.numpy(), causal=True)
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)


@pytest.mark.parametrize("Nq,Nk", [(17, 70), (6, 6), (9, 4)])
def test_fp32_queries_at_the_end(cuda_lib, Nq, Nk):
    q, k, v = si.attn_inputs(2, 2, Nq, Nk, 16, torch.float32, seed=500 + Nq + Nk)
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy(), causal=True)
    for tiles in (None, (4, 3)):
        if tiles is None:
            o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
        else:
            o, lse = cuda_lib.attn_fwd_f32_tiles(q.cuda(), k.cuda(), v.cuda(), *tiles, causal=True)
        _sync(cuda_lib)
        assert_lse_close(lse, rl)
        assert_out_close(o, ro, F32_ATTN_ATOL, lse_ref=rl)


@pytest.mark.parametrize("Nq", [8192, 4096])
def test_launch_dealt_in_phases_with_kv_len_and_grouped_heads(cuda_lib, Nq):
    # 64 MiB of K/V (B2 H_kv8 Nk8192 d128) exceeds what a phase of the dealing keeps in L2, so the
    # launch runs over bands of heads, with odd rounds reading key tiles top down; the second
    # sequence's cache ends at 5000 keys.  Square (Nq = Nk) and offset (Nq < Nk) causal; sampled rows.
    B, H, Hkv, Nk, d = 2, 16, 8, 8192, 128
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, Nq, Nk, d, torch.bfloat16, seed=500 + Nq)
    kv_len = [Nk, 5000]
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True,
                               kv_len=torch.tensor(kv_len, dtype=torch.int32).cuda())
    _sync(cuda_lib)
    rows_i = si.sample_rows(Nq, 48, seed=Nq + 1).numpy()
    flat = np.concatenate([(bh * Nq) + rows_i for bh in range(B * H)])
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True, kv_len=kv_len, rows=flat)
    assert_lse_close(lse.reshape(-1)[torch.from_numpy(flat).cuda()], rl)
    assert_out_close(o.reshape(-1, d)[torch.from_numpy(flat).cuda()], ro, BF16_O_ATOL, lse_ref=rl)
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()


@pytest.mark.slow
def test_full_size_chunked_prefill_grouped(cuda_lib):
    """The benchmarked chunked prefill: B8 H32 H_kv8, 2048 new queries against a 32768-key cache, d128,
    causal at the end; sampled query rows of four (b, h) against the oracle on their key/value head."""
    B, H, Hkv, Nq, Nk, d = 8, 32, 8, 2048, 32768, 128
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, Nq, Nk, d, torch.bfloat16, seed=0, device="cuda")
    o, lse = cuda_lib.attn_fwd(q, k, v, causal=True)
    _sync(cuda_lib)
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    rows = si.sample_rows(Nq, 48, seed=2).numpy()
    for b, h in ((0, 0), (3, 13), (5, 22), (B - 1, H - 1)):
        hk = h // (H // Hkv)
        ro, rl = oracle.attention(bf16_bits(q[b:b + 1, h:h + 1]), bf16_bits(k[b:b + 1, hk:hk + 1]),
                                  bf16_bits(v[b:b + 1, hk:hk + 1]), causal=True, rows=rows)
        assert_lse_close(lse[b, h][torch.from_numpy(rows).cuda()], rl)
        assert_out_close(o[b, h][torch.from_numpy(rows).cuda()], ro, BF16_O_ATOL)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq", [2, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_multi_token_decode(cuda_lib, d, Nq, causal):
    # a few new tokens per sequence against a grouped KV cache: the group's query heads x new tokens run
    # as the rows of one plane (each K/V row read once per group); causal: a row's position is its token
    B, H, Hkv, Nk = 3, 16, 4, 3000
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, Nq, Nk, d, torch.bfloat16, seed=600 + d + Nq)
    kv_len = [3000, 777, 0]
    kvd = torch.tensor(kv_len, dtype=torch.int32).cuda()
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, kv_len=kvd)
    _sync(cuda_lib)
    g = H // Hkv
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k.repeat_interleave(g, dim=1)),
                              bf16_bits(v.repeat_interleave(g, dim=1)), causal=causal, kv_len=kv_len)
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)
    if not causal:  # the split-KV entry point takes the same grouped path
        o2, lse2 = cuda_lib.attn_splitkv(q.cuda(), k.cuda(), v.cuda(), 8, kv_len=kvd)
        _sync(cuda_lib)
        assert_lse_close(lse2, rl)
        assert_out_close(o2, ro, BF16_O_ATOL, lse_ref=rl)


@pytest.mark.parametrize("H,Hkv,Nq", [(32, 2, 8), (32, 2, 9), (8, 1, 17)])
def test_grouped_decode_rows_at_and_past_128(cuda_lib, H, Hkv, Nq):
    # g * Nq = 128 rows fill a plane exactly; 144 rows take the one-item-per-query-head path
    B, Nk, d = 2, 700, 128
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, Nq, Nk, d, torch.bfloat16, seed=700 + Nq)
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    _sync(cuda_lib)
    g = H // Hkv
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k.repeat_interleave(g, dim=1)),
                              bf16_bits(v.repeat_interleave(g, dim=1)), causal=True)
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)
