"""GPU parity of the fused attention backward (oa_attn_bwd) against the fp64 oracle.

Inputs: Q, K, V, dO ~ N(0, 1) in bf16 (seeded); O and LSE come from this library's forward on the
same Q, K, V, as a training step passes them.  The oracle differentiates the exact attention of
the same bf16 values in fp64.

Tolerance, element by element, from the kernel's arithmetic (u = 2^-8, the unit roundoff of bf16's
8-bit significand).  The kernel rounds P and dS = P (dP - D) to bf16 before the tensor-core products;
D_i = dO_i . O_i uses the forward's bf16 O, which lies within 2u A_ic of the exact output,
A_ic = sum_j P_ij |V_jc|; all sums run in fp32 and the results are rounded to bf16 once.  To first order:
    dD_i  = 2u sum_c |dO_ic| A_ic                 (error of D_i)
    E_ij  = u |dS_ij| + P_ij dD_i                 (error of the bf16 dS_ij)
    |dV_j - ref| <= 2 (u sum_i P_ij |dO_i| + u |dV_j|)
    |dK_j - ref| <= 2 (scale sum_i E_ij |Q_i| + u |dK_j|)
    |dQ_i - ref| <= 2 (scale sum_j E_ij |K_j| + u |dQ_i|)
plus 1e-6 absolute; the factor 2 covers the fp32 sums and second-order terms.  P, dS and A are
computed here in fp64 for the bound only; the values compared against are the oracle's.
"""
import numpy as np
import pytest
import torch

import online_softmax_attention_tiled_gb300 as oa
import oracle
import synth_inputs as si
from parity import bf16_bits

pytestmark = pytest.mark.gpu

U = 2.0 ** -8
DEV = "cuda:0"


def _inputs(B, H, Nq, Nk, d, seed):
    q, k, v = si.attn_inputs(B, H, Nq, Nk, d, torch.bfloat16, seed=seed)
    do = si.randn((B, H, Nq, d), seed + 3, torch.bfloat16)
    return q, k, v, do


def _bounds(q, k, v, do, causal, scale, q_rows, k_rows, block=512):
    """First-order error bounds (before the output-rounding term) of one head: dq at q_rows, dk and dv
    at k_rows.  q, do [Nq, d], k, v [Nk, d] as fp64 CPU tensors."""
    Nq, d = q.shape
    Nk = k.shape[0]
    q_rows = torch.as_tensor(q_rows, dtype=torch.int64)
    k_rows = torch.as_tensor(k_rows, dtype=torch.int64)
    tq = torch.zeros(len(q_rows), d, dtype=torch.float64)
    tk = torch.zeros(len(k_rows), d, dtype=torch.float64)
    tv = torch.zeros(len(k_rows), d, dtype=torch.float64)
    aq, ak, av, ado = q.abs(), k.abs(), v.abs(), do.abs()
    for i0 in range(0, Nq, block):
        i1 = min(Nq, i0 + block)
        s = scale * (q[i0:i1] @ k.T)
        if causal:  # the queries are the last Nq positions: query i sees keys j <= i + Nk - Nq
            hide = torch.arange(Nk)[None, :] > torch.arange(i0, i1)[:, None] + (Nk - Nq)
            s = s.masked_fill(hide, float("-inf"))
        lse = torch.logsumexp(s, dim=1, keepdim=True)
        p = torch.where(torch.isfinite(lse), torch.exp(s - lse), torch.zeros_like(s))
        D = (do[i0:i1] * (p @ v)).sum(1, keepdim=True)
        ds = p * (do[i0:i1] @ v.T - D)
        dD = 2 * U * (ado[i0:i1] * (p @ av)).sum(1, keepdim=True)
        E = U * ds.abs() + p * dD
        sel = (q_rows >= i0) & (q_rows < i1)
        if sel.any():
            tq[sel] = scale * (E[q_rows[sel] - i0] @ ak)
        tk += scale * (E[:, k_rows].T @ aq[i0:i1])
        tv += U * (p[:, k_rows].T @ ado[i0:i1])
    return tq.numpy(), tk.numpy(), tv.numpy()


def _assert_within(got, ref, first_order, what):
    got = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else got
    assert not np.isnan(got).any(), f"{what}: NaN"
    tol = 2.0 * (first_order + U * np.abs(ref)) + 1e-6
    err = np.abs(got - ref)
    ratio = err / tol
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    print(f"{what}: max err/tol {ratio.max():.3f} (err {err.max():.3e}, max|ref| {np.abs(ref).max():.3e})")
    assert ratio.max() <= 1.0, (f"{what}: {(ratio > 1).sum()} elements beyond tolerance; worst at {worst}: "
                                f"{got[worst]!r} vs {ref[worst]!r} (tol {tol[worst]:.3e})")


def _run(q, k, v, do, causal, scale):
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = oa.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = oa.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return dq.cpu(), dk.cpu(), dv.cpu()


CASES = [
    # B, H, Nq, Nk, d, causal, scale (None = 1/sqrt(d))
    (1, 2, 300, 300, 64, True, None),
    (1, 2, 300, 300, 128, True, None),
    (2, 1, 200, 333, 64, False, None),
    (1, 1, 77, 500, 128, False, None),
    (1, 1, 513, 129, 64, False, None),
    (1, 1, 128, 128, 128, False, None),
    (1, 3, 129, 129, 64, True, None),
    (1, 1, 1, 1, 128, True, None),
    (1, 1, 256, 256, 64, False, 0.5),
    (2, 2, 384, 384, 128, True, None),
    # causal with more keys than queries (the queries at the end: chunked prefill against a cache)
    # and with fewer (the first Nq - Nk queries see no key)
    (1, 2, 200, 700, 64, True, None),
    (1, 2, 130, 517, 128, True, None),
    (1, 1, 300, 150, 64, True, None),
    (1, 1, 257, 100, 128, True, None),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,scale", CASES)
def test_attn_bwd_matches_oracle(B, H, Nq, Nk, d, causal, scale):
    seed = 40 + Nq + 7 * Nk + d
    q, k, v, do = _inputs(B, H, Nq, Nk, d, seed)
    sc = scale if scale is not None else 1.0 / np.sqrt(d)
    dq, dk, dv = _run(q, k, v, do, causal, sc)
    rq, rk, rv = oracle.attention_bwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), causal=causal,
                                      scale=sc)
    for b in range(B):
        for h in range(H):
            f64 = [t[b, h].to(torch.float64) for t in (q, k, v, do)]
            tq, tk, tv = _bounds(*f64, causal, sc, np.arange(Nq), np.arange(Nk))
            _assert_within(dq[b, h], rq[b, h], tq, f"dQ[{b},{h}]")
            _assert_within(dk[b, h], rk[b, h], tk, f"dK[{b},{h}]")
            _assert_within(dv[b, h], rv[b, h], tv, f"dV[{b},{h}]")


@pytest.mark.parametrize("B,H,Hkv,N,d,causal", [
    (1, 4, 2, 300, 128, True),
    (2, 8, 2, 200, 64, False),
    (1, 3, 1, 129, 64, True),
])
def test_attn_bwd_grouped_heads_match_oracle(B, H, Hkv, N, d, causal):
    # dK, dV of a key/value head sum over its query heads: their first-order bounds add up
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, N, N, d, torch.bfloat16, seed=60 + N)
    do = si.randn((B, H, N, d), 64 + N, torch.bfloat16)
    sc = 1.0 / np.sqrt(d)
    dq, dk, dv = _run(q, k, v, do, causal, sc)
    rq, rk, rv = oracle.attention_bwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), causal=causal,
                                      scale=sc)
    g = H // Hkv
    for b in range(B):
        for hk in range(Hkv):
            tk_sum, tv_sum = 0.0, 0.0
            for t in range(g):
                h = hk * g + t
                f64 = [x.to(torch.float64) for x in (q[b, h], k[b, hk], v[b, hk], do[b, h])]
                tq, tk, tv = _bounds(*f64, causal, sc, np.arange(N), np.arange(N))
                _assert_within(dq[b, h], rq[b, h], tq, f"dQ[{b},{h}]")
                tk_sum, tv_sum = tk_sum + tk, tv_sum + tv
            _assert_within(dk[b, hk], rk[b, hk], tk_sum, f"dK[{b},{hk}]")
            _assert_within(dv[b, hk], rv[b, hk], tv_sum, f"dV[{b},{hk}]")


def test_attn_bwd_single_key_has_no_score_gradient():
    # one key: every weight is 1 whatever the scores, so dQ and dK vanish and dV is the sum of dO
    q, k, v, do = _inputs(1, 2, 200, 1, 64, seed=5)
    dq, dk, dv = _run(q, k, v, do, False, 0.125)
    # D_i and dP_i are the same dot product summed in two orders: their difference is fp32 noise
    assert dq.abs().max().item() < 1e-3 and dk.abs().max().item() < 1e-2
    ref = do.to(torch.float64).sum(dim=2)
    err = (dv[:, :, 0].to(torch.float64) - ref).abs()
    assert (err <= 2 * U * (do.to(torch.float64).abs().sum(dim=2) + ref.abs()) + 1e-6).all()


def test_attn_bwd_is_repeatable_and_keeps_inputs():
    q, k, v, do = _inputs(1, 2, 260, 260, 128, seed=9)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = oa.attn_fwd(qd, kd, vd, causal=True)
    keep = [t.clone() for t in (qd, kd, vd, dod, o, lse)]
    ws = torch.full((oa.attn_bwd_workspace_bytes(1, 2, 260, 128),), 0xFF, dtype=torch.uint8, device=DEV)
    a = oa.attn_bwd(qd, kd, vd, o, lse, dod, causal=True, workspace=ws)
    a = [t.clone() for t in a]
    b = oa.attn_bwd(qd, kd, vd, o, lse, dod, causal=True, workspace=ws)  # workspace left dirty by the first
    torch.cuda.synchronize()
    # dK, dV: plain stores, bit-identical; dQ: fp32 atomics, equal up to the order of the additions
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2 * U * a[0].float().abs().max().item()
    for x, y in zip(keep, (qd, kd, vd, dod, o, lse)):
        assert torch.equal(x, y)


def test_attn_bwd_binding_rejects_bad_arguments():
    q, k, v, do = (t.to(DEV) for t in _inputs(1, 1, 64, 64, 64, seed=1))
    o, lse = oa.attn_fwd(q, k, v)
    with pytest.raises(oa.OAError):
        oa.attn_bwd(q, k, v, o, None, do)
    with pytest.raises(oa.OAError):
        oa.attn_bwd(q, k, v, o[:, :, :32], lse, do)
    with pytest.raises(oa.OAError):
        oa.attn_bwd(q.float(), k.float(), v.float(), o.float(), lse, do.float())
    with pytest.raises(oa.OAError):
        oa.attn_bwd(q, k[:, :, :63], v, o, lse, do, causal=True)  # k and v of different lengths


def test_attn_bwd_full_size_sampled_rows():
    # causal B=1 H=32 N=8192 d=128 (the benchmarked backward): every gradient finite, and two heads
    # checked at sampled rows (both sides of every tile boundary, plus seeded fill) against the
    # row-sampled oracle, which needs no [N, N] matrix
    B, H, N, d = 1, 32, 8192, 128
    sc = 1.0 / np.sqrt(d)
    q, k, v, do = _inputs(B, H, N, N, d, seed=77)
    dq, dk, dv = _run(q, k, v, do, True, sc)
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    rows = si.sample_rows(N, 192, seed=3).numpy()
    for h in (0, H - 1):
        rq, rk, rv = oracle.attention_bwd_sampled(*(bf16_bits(t[0, h]) for t in (q, k, v, do)), rows, rows,
                                                  causal=True, scale=sc)
        tq, tk, tv = _bounds(*(t[0, h].to(torch.float64) for t in (q, k, v, do)), True, sc, rows, rows)
        _assert_within(dq[0, h][rows], rq, tq, f"dQ[0,{h}] sampled")
        _assert_within(dk[0, h][rows], rk, tk, f"dK[0,{h}] sampled")
        _assert_within(dv[0, h][rows], rv, tv, f"dV[0,{h}] sampled")


def test_attn_bwd_full_size_d64_sampled_rows():
    # non-causal B=4 H=16 N=4096 d=64 (32 query tiles stream through each key-tile CTA, wrapping
    # the d = 64 kernel's three-stage ring many times): every gradient finite, and two heads checked
    # at sampled rows against the row-sampled oracle
    B, H, N, d = 4, 16, 4096, 64
    sc = 1.0 / np.sqrt(d)
    q, k, v, do = _inputs(B, H, N, N, d, seed=91)
    dq, dk, dv = _run(q, k, v, do, False, sc)
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    rows = si.sample_rows(N, 160, seed=5).numpy()
    for b, h in ((0, 0), (B - 1, H - 1)):
        rq, rk, rv = oracle.attention_bwd_sampled(*(bf16_bits(t[b, h]) for t in (q, k, v, do)), rows, rows,
                                                  causal=False, scale=sc)
        tq, tk, tv = _bounds(*(t[b, h].to(torch.float64) for t in (q, k, v, do)), False, sc, rows, rows)
        _assert_within(dq[b, h][rows], rq, tq, f"dQ[{b},{h}] sampled")
        _assert_within(dk[b, h][rows], rk, tk, f"dK[{b},{h}] sampled")
        _assert_within(dv[b, h][rows], rv, tv, f"dV[{b},{h}] sampled")


@pytest.mark.parametrize("lq,lk,H,Hkv,d,causal", [
    ([300, 129, 1, 257], [300, 129, 1, 257], 4, 2, 128, True),
    ([100, 0, 200, 64, 33], [150, 80, 0, 64, 200], 2, 2, 64, False),
    ([130, 70], [200, 70], 4, 1, 128, True),   # causal with more keys than queries
    ([60, 300, 200], [500, 300, 90], 2, 1, 64, True),  # more keys, equal, fewer keys (bottom-right)
    ([700, 300, 1], [700, 300, 1], 4, 2, 64, True),  # d = 64, packed, several steps per CTA
])
def test_attn_bwd_varlen_matches_oracle(lq, lk, H, Hkv, d, causal):
    q, k, v, cq, ck = si.varlen_inputs(lq, lk, H, Hkv, d, torch.bfloat16, seed=80 + sum(lq))
    do = si.randn(tuple(q.shape), 90 + sum(lq), torch.bfloat16)
    sc = 1.0 / np.sqrt(d)
    qd, kd, vd, dod, cqd, ckd = (t.to(DEV) for t in (q, k, v, do, cq, ck))
    o, lse = oa.attn_fwd_varlen(qd, kd, vd, cqd, ckd, max(lq), max(lk), causal=causal, scale=sc)
    dq, dk, dv = oa.attn_bwd_varlen(qd, kd, vd, o, lse, dod, cqd, ckd, max(lq), max(lk), causal=causal, scale=sc)
    oa.sync_status()
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    rq, rk, rv = oracle.attention_bwd_varlen(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), cq.numpy(),
                                             ck.numpy(), causal=causal, scale=sc)
    g = H // Hkv
    for s in range(len(lq)):
        sq, sk = slice(int(cq[s]), int(cq[s + 1])), slice(int(ck[s]), int(ck[s + 1]))
        if lq[s] == 0 or lk[s] == 0:  # no query or no key: the gradients there are exactly zero
            assert torch.all(dq[sq] == 0) and torch.all(dk[sk] == 0) and torch.all(dv[sk] == 0)
            continue
        for hk in range(Hkv):
            tk_sum, tv_sum = 0.0, 0.0
            for t in range(g):
                h = hk * g + t
                f64 = [x.to(torch.float64) for x in (q[sq, h], k[sk, hk], v[sk, hk], do[sq, h])]
                tq, tk, tv = _bounds(*f64, causal, sc, np.arange(lq[s]), np.arange(lk[s]))
                _assert_within(dq[sq, h], rq[sq, h], tq, f"dQ seq {s} head {h}")
                tk_sum, tv_sum = tk_sum + tk, tv_sum + tv
            _assert_within(dk[sk, hk], rk[sk, hk], tk_sum, f"dK seq {s} head {hk}")
            _assert_within(dv[sk, hk], rv[sk, hk], tv_sum, f"dV seq {s} head {hk}")


def test_attn_bwd_varlen_reports_a_key_sequence_longer_than_declared():
    lq = lk = [200, 300]
    q, k, v, cq, ck = si.varlen_inputs(lq, lk, 2, 2, 64, torch.bfloat16, seed=3)
    qd, kd, vd, cqd, ckd = (t.to(DEV) for t in (q, k, v, cq, ck))
    o, lse = oa.attn_fwd_varlen(qd, kd, vd, cqd, ckd, 300, 300)
    oa.attn_bwd_varlen(qd, kd, vd, o, lse, torch.ones_like(qd), cqd, ckd, 300, 256)  # 300 keys > 256 declared
    with pytest.raises(oa.OAError) as e:
        oa.sync_status()
    assert e.value.status == oa.OA_ERR_INVALID
    oa.sync_status()  # cleared


def test_attn_bwd_full_size_grouped_heads_sampled_rows():
    # causal B=1 H=32 H_kv=8 N=8192 d=128 (the benchmarked grouped backward): dK, dV of two key/value
    # heads at sampled rows are the sums of the row-sampled oracle over each group's four query heads
    B, H, Hkv, N, d = 1, 32, 8, 8192, 128
    sc = 1.0 / np.sqrt(d)
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, N, N, d, torch.bfloat16, seed=79)
    do = si.randn((B, H, N, d), 82, torch.bfloat16)
    dq, dk, dv = _run(q, k, v, do, True, sc)
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    rows = si.sample_rows(N, 96, seed=5).numpy()
    g = H // Hkv
    for hk in (0, Hkv - 1):
        sum_k, sum_v, tk_sum, tv_sum = 0.0, 0.0, 0.0, 0.0
        for t in range(g):
            h = hk * g + t
            rq, rk, rv = oracle.attention_bwd_sampled(*(bf16_bits(x[0, i]) for x, i in
                                                        ((q, h), (k, hk), (v, hk), (do, h))), rows, rows,
                                                      causal=True, scale=sc)
            tq, tk, tv = _bounds(*(x[0, i].to(torch.float64) for x, i in ((q, h), (k, hk), (v, hk), (do, h))),
                                 True, sc, rows, rows)
            _assert_within(dq[0, h][rows], rq, tq, f"dQ[0,{h}] sampled")
            sum_k, sum_v, tk_sum, tv_sum = sum_k + rk, sum_v + rv, tk_sum + tk, tv_sum + tv
        _assert_within(dk[0, hk][rows], sum_k, tk_sum, f"dK[0,{hk}] sampled")
        _assert_within(dv[0, hk][rows], sum_v, tv_sum, f"dV[0,{hk}] sampled")
