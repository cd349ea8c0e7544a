"""Grouped key/value heads and packed variable-length sequences vs the fp64 oracle (gpu).

Covers the tensor-core forward (oa_attn_fwd_gqa, oa_attn_fwd_varlen), the fp32 forward with grouped
heads and split-KV decode over a grouped KV cache (oa_attn_splitkv_gqa).
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import BF16_O_ATOL, assert_lse_close, assert_out_close, bf16_bits

pytestmark = pytest.mark.gpu


def _sync(oa):
    torch.cuda.synchronize()
    oa.sync_status()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hkv", [1, 2, 4])
def test_gqa_tensor_core(cuda_lib, d, causal, Hkv):
    B, H, N = 2, 8, 300
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, N, N, d, torch.bfloat16, seed=40 + d + Hkv)
    kv_len = [N, 129]
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal,
                               kv_len=torch.tensor(kv_len, dtype=torch.int32).cuda())
    _sync(cuda_lib)
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=causal, kv_len=kv_len)
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)


def test_gqa_fp32(cuda_lib):
    B, H, Hkv, Nq, Nk, d = 2, 6, 3, 33, 70, 40
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, Nq, Nk, d, torch.float32, seed=50)
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda())
    _sync(cuda_lib)
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, 1e-5, lse_ref=rl)


def test_gqa_rejects_non_divisor(cuda_lib):
    q, k, v = si.attn_inputs_gqa(1, 6, 4, 16, 16, 64, torch.bfloat16, seed=1)
    with pytest.raises(cuda_lib.OAError):
        cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda())


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_gqa_splitkv_decode(cuda_lib, dtype, d):
    # a grouped KV cache of different lengths per sequence, one query token per head
    B, H, Hkv, Nk, splits = 4, 8, 2, 1000, 8
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, 1, Nk, d, dtype, seed=60 + d)
    kv_len = [1000, 1, 0, 555]
    o, lse = cuda_lib.attn_splitkv(q.cuda(), k.cuda(), v.cuda(), splits,
                                   kv_len=torch.tensor(kv_len, dtype=torch.int32).cuda())
    _sync(cuda_lib)
    if dtype == torch.bfloat16:
        ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), kv_len=kv_len)
        atol = BF16_O_ATOL
    else:
        ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy(), kv_len=kv_len)
        atol = 2e-5
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, atol, lse_ref=rl)


@pytest.mark.parametrize("H,Hkv", [(16, 8), (16, 4), (16, 2), (16, 1)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nq", [1, 2])
def test_gqa_decode_groups(cuda_lib, H, Hkv, d, nq):
    # one or two queries per head run each group's (head, query) pairs as the rows of one plane (forward
    # kernel); both entry points, every group size, against the oracle
    B, Nk = 3, 700
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, nq, Nk, d, torch.bfloat16, seed=70 + H // Hkv + d + nq)
    kv_len = [700, 129, 0]
    kvd = torch.tensor(kv_len, dtype=torch.int32).cuda()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), kv_len=kv_len)
    o, lse = cuda_lib.attn_splitkv(q.cuda(), k.cuda(), v.cuda(), 6, kv_len=kvd)
    _sync(cuda_lib)
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)
    o2, lse2 = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), kv_len=kvd)
    _sync(cuda_lib)
    assert_lse_close(lse2, rl)
    assert_out_close(o2, ro, BF16_O_ATOL, lse_ref=rl)


@pytest.mark.parametrize("H,Hkv,nq", [(16, 2, 20), (8, 2, 40), (16, 4, 33)])
def test_gqa_splitkv_group_kernel(cuda_lib, H, Hkv, nq):
    # more than 128 (head, query) rows per group: split-KV takes its group kernel (each K/V row read once
    # and scored against every query of the group, chunks merged by LSE)
    B, Nk, d = 2, 1500, 128
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, nq, Nk, d, torch.bfloat16, seed=80 + nq)
    kv_len = [1500, 611]
    kvd = torch.tensor(kv_len, dtype=torch.int32).cuda()
    g = H // Hkv
    assert g * nq > 128
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k.repeat_interleave(g, dim=1)),
                              bf16_bits(v.repeat_interleave(g, dim=1)), kv_len=kv_len)
    o, lse = cuda_lib.attn_splitkv(q.cuda(), k.cuda(), v.cuda(), 12, kv_len=kvd)
    _sync(cuda_lib)
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)


def _varlen_check(oa, lq, lk, H, Hkv, d, causal, seed, max_q=None, max_k=None):
    q, k, v, cq, ck = si.varlen_inputs(lq, lk, H, Hkv, d, torch.bfloat16, seed=seed)
    o, lse = oa.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(),
                                max(lq) if max_q is None else max_q, max(lk) if max_k is None else max_k,
                                causal=causal)
    _sync(oa)
    ro, rl = oracle.attention_varlen(bf16_bits(q), bf16_bits(k), bf16_bits(v), cq.numpy(), ck.numpy(),
                                     causal=causal)
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_self_attention(cuda_lib, d, causal):
    # lengths crossing tile edges, a 1-token and an empty sequence, one over two tiles of 256 rows
    lens = [300, 1, 0, 513, 128, 77, 256, 129]
    _varlen_check(cuda_lib, lens, lens, 4, 2, d, causal, seed=70 + d)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_cross_lengths(cuda_lib, causal):
    # query and key lengths differ per sequence (a sequence with keys but no queries, and one with
    # queries but no keys: O = 0, lse = -inf)
    lq = [100, 0, 257, 40, 3]
    lk = [333, 50, 129, 0, 700]
    _varlen_check(cuda_lib, lq, lk, 8, 8, 128, causal, seed=80)


def test_varlen_many_sequences(cuda_lib):
    # more work items than SMs: 64 sequences x 8 heads, lengths in [0, 600]
    lens = si.varlen_lengths(64, 600, seed=90)
    _varlen_check(cuda_lib, lens, lens, 8, 2, 64, True, seed=91)


def test_varlen_sequence_longer_than_declared_max(cuda_lib):
    # a query sequence longer than max_seqlen_q is reported through the status word; the kernel
    # writes the rows it covers and reads or writes nothing outside the tensors
    lens = [600, 100]
    q, k, v, cq, ck = si.varlen_inputs(lens, lens, 2, 2, 64, torch.bfloat16, seed=95)
    cuda_lib.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), 300, 600)
    torch.cuda.synchronize()
    with pytest.raises(cuda_lib.OAError):
        cuda_lib.sync_status()
    cuda_lib.sync_status()  # the word was cleared: the next call is clean


@pytest.mark.slow
def test_full_size_decode_grouped_cache(cuda_lib):
    """The benchmarked grouped decode: B32 H32 H_kv8 Nq1 Nk32768 d128 bf16, 64 chunks of 512, the same
    truncated sequences; sampled (b, h) rows against the oracle on their key/value head."""
    B, H, Hkv, Nk, d = 32, 32, 8, 32768, 128
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, 1, Nk, d, torch.bfloat16, seed=0, device="cuda")
    kv_len = si.decode_kv_len(B, Nk, seed=0)
    o, lse = cuda_lib.attn_splitkv(q, k, v, 64, kv_len=kv_len.cuda())
    _sync(cuda_lib)
    trunc = torch.nonzero(kv_len < Nk).reshape(-1).tolist()
    for b in sorted(set([0, B - 1] + trunc + list(range(3, B, 9)))):
        n = int(kv_len[b])
        for h in (0, 5, H - 1):
            hk = h // (H // Hkv)
            ro, rl = oracle.attention(bf16_bits(q[b:b + 1, h:h + 1]), bf16_bits(k[b:b + 1, hk:hk + 1, :n]),
                                      bf16_bits(v[b:b + 1, hk:hk + 1, :n]))
            assert_lse_close(lse[b, h], rl)
            assert_out_close(o[b, h], ro[0, 0], BF16_O_ATOL)
    assert not torch.isnan(o).any()


@pytest.mark.slow
def test_full_size_varlen_causal_grouped(cuda_lib):
    """The benchmarked packed prefill: 16 causal sequences of U[1024, 8192] tokens, H32 H_kv8 d128;
    sampled rows (both sides of every tile boundary) of three sequences and two heads."""
    H, Hkv, d = 32, 8, 128
    lens = si.varlen_lengths(16, 8192, seed=0, min_len=1024)
    q, k, v, cq, ck = si.varlen_inputs(lens, lens, H, Hkv, d, torch.bfloat16, seed=0)
    o, lse = cuda_lib.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), max(lens), max(lens),
                                      causal=True)
    _sync(cuda_lib)
    o, lse = o.cpu(), lse.cpu()
    for s in (0, 7, len(lens) - 1):
        L, a = lens[s], int(cq[s])
        rows = si.sample_rows(L, 64, seed=s)
        for h in (0, H - 1):
            hk = h // (H // Hkv)
            qs = q[a:a + L, h].reshape(1, 1, L, d)
            ks, vs = k[a:a + L, hk].reshape(1, 1, L, d), v[a:a + L, hk].reshape(1, 1, L, d)
            ro, rl = oracle.attention(bf16_bits(qs), bf16_bits(ks), bf16_bits(vs), causal=True, rows=rows.numpy())
            assert_lse_close(lse[a + rows, h], rl)
            assert_out_close(o[a + rows, h], ro, BF16_O_ATOL)
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()


@pytest.mark.parametrize("lens", [
    [4096] * 16,                                          # equal lengths
    [8192] + [512] * 15,                                  # one long sequence among short ones
    "bench",                                              # the benchmarked U[1024, 8192] lengths
])
def test_packed_causal_dealt_in_phases_covers_every_row(cuda_lib, lens):
    """Packed causal launches whose K/V exceeds L2 pick their phase count in the kernel from the
    sequence lengths; whatever it picks, every row of every sequence and head must come out.  Each
    sequence is also run alone through the dense path (another instance and dealing) and every row
    compared; a few rows per sequence against the oracle."""
    if lens == "bench":
        lens = si.varlen_lengths(16, 8192, seed=0, min_len=1024)
    H, Hkv, d = 32, 8, 128
    q, k, v, cq, ck = si.varlen_inputs(lens, lens, H, Hkv, d, torch.bfloat16, seed=len(lens) + max(lens))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = cuda_lib.attn_fwd_varlen(qd, kd, vd, cq.cuda(), ck.cuda(), max(lens), max(lens), causal=True)
    _sync(cuda_lib)
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    for s_, L in enumerate(lens):
        a = int(cq[s_])
        qs = qd[a:a + L].permute(1, 0, 2).unsqueeze(0).contiguous()
        ks = kd[a:a + L].permute(1, 0, 2).unsqueeze(0).contiguous()
        vs = vd[a:a + L].permute(1, 0, 2).unsqueeze(0).contiguous()
        od, ld = cuda_lib.attn_fwd(qs, ks, vs, causal=True)
        _sync(cuda_lib)
        # the same rows through another dealing: equal up to the order of the key tiles
        assert torch.allclose(lse[a:a + L].t().float(), ld[0].float(), atol=1e-3, rtol=0), s_
        assert (o[a:a + L].permute(1, 0, 2).float() - od[0].float()).abs().max().item() <= BF16_O_ATOL, s_
        if s_ % 5 == 0:
            rows = si.sample_rows(L, 16, seed=s_)
            h = s_ % H
            hk = h // (H // Hkv)
            ro, rl = oracle.attention(bf16_bits(q[a:a + L, h].reshape(1, 1, L, d)),
                                      bf16_bits(k[a:a + L, hk].reshape(1, 1, L, d)),
                                      bf16_bits(v[a:a + L, hk].reshape(1, 1, L, d)), causal=True, rows=rows.numpy())
            assert_lse_close(lse[a + rows, h].cpu(), rl)
            assert_out_close(o[a + rows, h].cpu(), ro, BF16_O_ATOL)
