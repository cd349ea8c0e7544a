"""Seeded random sweep of the bf16 forward, the backward and the row softmax against the fp64 oracle (gpu).

The hand-picked cases of the other files pin each feature; here fixed pseudo-random draws combine
them -- batch, query and key/value heads (grouping), query and key lengths (ragged against the
128-row and 128-key tiles, more queries than keys, single rows), head size, causality, per-sequence
key lengths including empty ones, softmax widths across the one-CTA, cluster and streaming paths --
so that combinations nobody wrote down get checked too; likewise packed sequences (lengths from 0,
queries and keys of different lengths), split-KV decode over grouped caches with per-sequence
lengths, and the fp32 forward with random tiles.  Every draw is a deterministic function of its
case number.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import BF16_O_ATOL, assert_lse_close, assert_out_close, assert_softmax_close, bf16_bits

pytestmark = pytest.mark.gpu


def _fwd_case(n):
    r = np.random.default_rng(1000 + n)
    d = int(r.choice([64, 128]))
    hkv = int(r.choice([1, 2, 3]))
    g = int(r.choice([1, 2, 4]))
    B = int(r.integers(1, 4))
    Nq = int(r.choice([1, 2, 7, 64, 127, 128, 129, 200, 256, 257, 383, 511]))
    Nk = int(r.choice([1, 5, 100, 128, 129, 300, 513, 700])) if r.random() < 0.6 else Nq
    causal = bool(r.random() < 0.6)
    kv_len = None
    if r.random() < 0.4:
        kv_len = [int(x) for x in r.integers(0, Nk + 1, size=B)]
    return B, hkv * g, hkv, Nq, Nk, d, causal, kv_len


@pytest.mark.parametrize("n", range(64))
def test_forward_sweep(cuda_lib, n):
    B, H, Hkv, Nq, Nk, d, causal, kv_len = _fwd_case(n)
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, Nq, Nk, d, torch.bfloat16, seed=2000 + n)
    kvd = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32).cuda()
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, kv_len=kvd)
    torch.cuda.synchronize()
    cuda_lib.sync_status()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=causal, kv_len=kv_len)
    assert_lse_close(lse, rl, what=f"lse case {n}")
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)


@pytest.mark.parametrize("n", range(16))
def test_backward_sweep(cuda_lib, n):
    # held to the per-element bound of the backward tests (first-order error of the bf16 roundings of
    # P, dS and the outputs; summed over a group's query heads for dK, dV)
    from test_gpu_attn_bwd import _assert_within, _bounds

    r = np.random.default_rng(3000 + n)
    d = int(r.choice([64, 128]))
    hkv = int(r.choice([1, 2]))
    g = int(r.choice([1, 2]))
    H = hkv * g
    Nq = int(r.choice([64, 129, 200, 300]))
    Nk = int(r.choice([64, 129, 250, 400])) if r.random() < 0.5 else Nq
    causal = bool(r.random() < 0.6)
    sc = 1.0 / math.sqrt(d)
    q, k, v = si.attn_inputs_gqa(1, H, hkv, Nq, Nk, d, torch.bfloat16, seed=4000 + n)
    do = si.randn((1, H, Nq, d), 5000 + n, torch.bfloat16)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = cuda_lib.attn_fwd(qc, kc, vc, causal=causal)
    dq, dk, dv = cuda_lib.attn_bwd(qc, kc, vc, o, lse, doc, causal=causal)
    torch.cuda.synchronize()
    cuda_lib.sync_status()
    rq, rk, rv = oracle.attention_bwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), causal=causal,
                                      scale=sc)
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    for hk in range(hkv):
        tk_sum, tv_sum = 0.0, 0.0
        for t in range(g):
            h = hk * g + t
            f64 = [x.to(torch.float64) for x in (q[0, h], k[0, hk], v[0, hk], do[0, h])]
            tq, tk, tv = _bounds(*f64, causal, sc, np.arange(Nq), np.arange(Nk))
            _assert_within(dq[0, h], rq[0, h], tq, f"dQ[{h}] case {n}")
            tk_sum, tv_sum = tk_sum + tk, tv_sum + tv
        _assert_within(dk[0, hk], rk[0, hk], tk_sum, f"dK[{hk}] case {n}")
        _assert_within(dv[0, hk], rv[0, hk], tv_sum, f"dV[{hk}] case {n}")


@pytest.mark.parametrize("n", range(24))
def test_softmax_sweep(cuda_lib, n):
    r = np.random.default_rng(6000 + n)
    cols = int(r.choice([1, 3, 31, 257, 1023, 2049, 4097, 9000, 33000, 65537, 70000, 140000]))
    rows = int(r.integers(1, 9))
    x = si.softmax_input(rows, cols, seed=7000 + n)[0]
    unaligned = bool(r.random() < 0.3)
    if unaligned:  # a column slice: rows start off the 16-byte grid (the scalar path)
        big = torch.empty(rows, cols + 3)
        big[:, 1:cols + 1] = x
        xd = big.cuda()[:, 1:cols + 1]
    else:
        xd = x.cuda()
    y, lse = cuda_lib.softmax_rows(xd)
    torch.cuda.synchronize()
    cuda_lib.sync_status()
    ry, rl = oracle.softmax_rows(x.numpy())
    assert_softmax_close(y, ry, what=f"y case {n} ({rows}x{cols}{' unaligned' if unaligned else ''})")
    assert_lse_close(lse, rl, what=f"lse case {n}")


@pytest.mark.parametrize("n", range(16))
def test_packed_forward_sweep(cuda_lib, n):
    r = np.random.default_rng(8000 + n)
    d = int(r.choice([64, 128]))
    hkv = int(r.choice([1, 2]))
    H = hkv * int(r.choice([1, 2, 4]))
    S = int(r.integers(1, 7))
    lq = [int(x) for x in r.choice([0, 1, 3, 64, 127, 128, 129, 300, 513], size=S)]
    same = r.random() < 0.5
    lk = list(lq) if same else [int(x) for x in r.choice([0, 1, 5, 100, 129, 256, 400, 700], size=S)]
    if sum(lq) == 0:
        lq[0] = 1
    if sum(lk) == 0:
        lk[-1] = 1
    causal = bool(r.random() < 0.6)
    q, k, v, cq, ck = si.varlen_inputs(lq, lk, H, hkv, d, torch.bfloat16, seed=9000 + n)
    o, lse = cuda_lib.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), max(max(lq), 1),
                                      max(max(lk), 1), causal=causal)
    torch.cuda.synchronize()
    cuda_lib.sync_status()
    ro, rl = oracle.attention_varlen(bf16_bits(q), bf16_bits(k), bf16_bits(v), cq.numpy(), ck.numpy(), causal=causal)
    assert_lse_close(lse, rl, what=f"lse case {n} (lq {lq}, lk {lk}, H{H}/{hkv}, d{d}, causal {causal})")
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)


@pytest.mark.parametrize("n", range(12))
def test_splitkv_sweep(cuda_lib, n):
    r = np.random.default_rng(10000 + n)
    d = int(r.choice([64, 128]))
    hkv = int(r.choice([1, 2, 4]))
    H = hkv * int(r.choice([1, 2, 4]))
    B = int(r.integers(1, 5))
    Nq = int(r.choice([1, 1, 2, 5]))
    Nk = int(r.choice([1, 37, 512, 1000, 3000]))
    splits = int(r.choice([1, 2, 7, 16, 64]))
    kv_len = [int(x) for x in r.integers(0, Nk + 1, size=B)] if r.random() < 0.5 else None
    q, k, v = si.attn_inputs_gqa(B, H, hkv, Nq, Nk, d, torch.bfloat16, seed=11000 + n)
    kvd = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32).cuda()
    o, lse = cuda_lib.attn_splitkv(q.cuda(), k.cuda(), v.cuda(), splits, kv_len=kvd)
    torch.cuda.synchronize()
    cuda_lib.sync_status()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), kv_len=kv_len)
    what = f"case {n} (B{B} H{H}/{hkv} {Nq}x{Nk} d{d} splits {splits} kv_len {kv_len})"
    assert_lse_close(lse, rl, what=f"lse {what}")
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)


@pytest.mark.parametrize("n", range(8))
def test_fp32_forward_sweep(cuda_lib, n):
    from parity import F32_ATTN_ATOL

    r = np.random.default_rng(12000 + n)
    d = int(r.choice([4, 16, 32, 64]))
    Nq = int(r.choice([1, 6, 37, 100]))
    Nk = int(r.choice([1, 3, 37, 129])) if r.random() < 0.5 else Nq
    causal = bool(r.random() < 0.5)
    Br, Bc = int(r.integers(1, 65)), int(r.integers(1, 65))
    q, k, v = si.attn_inputs(2, 2, Nq, Nk, d, torch.float32, seed=13000 + n)
    o, lse = cuda_lib.attn_fwd_f32_tiles(q.cuda(), k.cuda(), v.cuda(), Br, Bc, causal=causal)
    torch.cuda.synchronize()
    cuda_lib.sync_status()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy(), causal=causal)
    assert_lse_close(lse, rl, what=f"lse case {n} ({Nq}x{Nk} d{d} Br{Br} Bc{Bc} causal {causal})")
    assert_out_close(o, ro, F32_ATTN_ATOL, lse_ref=rl)


@pytest.mark.parametrize("n", range(10))
def test_packed_backward_sweep(cuda_lib, n):
    from test_gpu_attn_bwd import _assert_within, _bounds

    r = np.random.default_rng(14000 + n)
    d = int(r.choice([64, 128]))
    hkv = int(r.choice([1, 2]))
    g = int(r.choice([1, 2]))
    H = hkv * g
    S = int(r.integers(1, 5))
    lq = [int(x) for x in r.choice([0, 1, 64, 129, 200, 300], size=S)]
    lk = list(lq) if r.random() < 0.5 else [int(x) for x in r.choice([0, 1, 100, 129, 250], size=S)]
    if sum(lq) == 0:
        lq[0] = 1
    if sum(lk) == 0:
        lk[-1] = 1
    causal = bool(r.random() < 0.6)
    sc = 1.0 / math.sqrt(d)
    q, k, v, cq, ck = si.varlen_inputs(lq, lk, H, hkv, d, torch.bfloat16, seed=15000 + n)
    do = si.randn(tuple(q.shape), 16000 + n, torch.bfloat16)
    qd, kd, vd, dod, cqd, ckd = (t.cuda() for t in (q, k, v, do, cq, ck))
    mq, mk = max(max(lq), 1), max(max(lk), 1)
    o, lse = cuda_lib.attn_fwd_varlen(qd, kd, vd, cqd, ckd, mq, mk, causal=causal, scale=sc)
    dq, dk, dv = cuda_lib.attn_bwd_varlen(qd, kd, vd, o, lse, dod, cqd, ckd, mq, mk, causal=causal, scale=sc)
    torch.cuda.synchronize()
    cuda_lib.sync_status()
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    rq, rk, rv = oracle.attention_bwd_varlen(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), cq.numpy(),
                                             ck.numpy(), causal=causal, scale=sc)
    for s in range(S):
        sq, sk = slice(int(cq[s]), int(cq[s + 1])), slice(int(ck[s]), int(ck[s + 1]))
        if lq[s] == 0 or lk[s] == 0:  # no query or no key: the gradients there are exactly zero
            assert torch.all(dq[sq] == 0) and torch.all(dk[sk] == 0) and torch.all(dv[sk] == 0), f"case {n} seq {s}"
            continue
        for hk in range(hkv):
            tk_sum, tv_sum = 0.0, 0.0
            for t in range(g):
                h = hk * g + t
                f64 = [x.to(torch.float64) for x in (q[sq, h], k[sk, hk], v[sk, hk], do[sq, h])]
                tq, tk, tv = _bounds(*f64, causal, sc, np.arange(lq[s]), np.arange(lk[s]))
                _assert_within(dq[sq, h], rq[sq, h], tq, f"dQ case {n} seq {s} head {h}")
                tk_sum, tv_sum = tk_sum + tk, tv_sum + tv
            _assert_within(dk[sk, hk], rk[sk, hk], tk_sum, f"dK case {n} seq {s} head {hk}")
            _assert_within(dv[sk, hk], rv[sk, hk], tv_sum, f"dV case {n} seq {s} head {hk}")
