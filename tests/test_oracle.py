"""Pins for the CPU oracle: it must agree with something other than itself.

Each test ties one oracle function to values printed on the pages
(tests/golden/), to a closed form, to an invariant the pages state, to brute
force on a tiny input, or to an fp64 library routine.  Chosen so that a dropped
term, a wrong sign or index, a missing scale or a transposed operand in the
oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth_inputs as si

GOLD = os.path.join(os.path.dirname(__file__), "golden")
NEG_INF = float("-inf")


def golden(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# Worked examples printed on the pages
# ---------------------------------------------------------------------------

def test_roadmap_worked_example_offline():
    """Roadmap page s.3: x=[1,3,2] -> exps, sum and y as printed (4 decimals)."""
    g = golden("roadmap_s3_worked_example.json")
    half_ulp = 0.5 * 10 ** -g["printed_decimals"]
    y, lse = oracle.softmax_rows(np.array([g["x"]]))
    assert np.all(np.abs(y[0] - np.array(g["y"])) <= half_ulp)
    total = math.exp(lse[0] - g["max"])  # the sum of exp(x - max)
    assert abs(total - g["sum"]) <= half_ulp
    assert np.all(np.abs(y[0] * total - np.array(g["exponents"])) <= half_ulp)


def test_roadmap_worked_example_online_steps():
    """Roadmap page s.3: the running (m_k, d_k) after each element, as printed."""
    g = golden("roadmap_s3_worked_example.json")
    half_ulp = 0.5 * 10 ** -g["printed_decimals"]
    ms, ls = oracle.online_stats_trace(g["x"])
    for step, m, l in zip(g["online_steps"], ms, ls):
        assert m == step["m"]
        assert abs(l - step["d"]) <= half_ulp


def test_lesson_step1_stats_and_softmax():
    """Interview lesson Step 1: [1,3,2,5] -> m = 5, l = 1.2034379904932107 (1e-6); y == torch.softmax."""
    g = golden("lesson_step1_stats.json")
    m, l = oracle.online_stats(g["x"])
    assert m == g["m"]
    assert abs(l - g["l"]) < g["l_tolerance"]
    y, lse = oracle.softmax_rows(np.array([g["x"]]))
    ref = torch.softmax(torch.tensor(g["x"], dtype=torch.float64), 0).numpy()
    np.testing.assert_allclose(y[0], ref, rtol=1e-13, atol=0)
    # the scan's (m, l) and the three-pass lse describe the same normaliser
    assert abs((m + math.log(l)) - lse[0]) < 1e-14


def test_offline_equals_online_suggested_example():
    """Page 'Online softmax in attention', closing suggestion: x = [1, 5, 3] -- the
    incremental (m, s) must match the two/three-pass result to rounding noise."""
    x = [1.0, 5.0, 3.0]
    m, l = oracle.online_stats(x)
    y, lse = oracle.softmax_rows(np.array([x]))
    assert m == 5.0
    assert abs(m + math.log(l) - lse[0]) < 1e-15
    # closed form of the normaliser referred to the max: 1 + e^-2 + e^-4
    assert abs(l - (1.0 + math.exp(-2.0) + math.exp(-4.0))) < 1e-15


# ---------------------------------------------------------------------------
# The lesson's chunking / merge-order asserts (Step 1)
# ---------------------------------------------------------------------------

def _lesson_chunks(X):
    widths = golden("lesson_step1_stats.json")["chunk_widths"]
    out, c0 = [], 0
    for w in widths:
        out.append(X[:, c0:c0 + w])
        c0 += w
    assert c0 == X.shape[1]
    return out


def test_lesson_merge_order_invariance():
    """Any chunking and any merge order: left fold == tree == direct logsumexp;
    the fully masked row keeps l == 0, m == -inf, and nothing is NaN."""
    g = golden("lesson_step1_stats.json")
    X = si.lesson_matrix(seed=0).double().numpy()
    assert X.shape == tuple(g["matrix_shape"])
    chunks = _lesson_chunks(X)
    stats = [[oracle.online_stats(c[r]) for r in range(X.shape[0])] for c in chunks]
    ref = torch.logsumexp(torch.from_numpy(X), -1).numpy()
    _, lse_def = oracle.softmax_rows(X)
    for r in range(X.shape[0]):
        m_f, l_f = stats[0][r]
        for c in range(1, len(chunks)):
            m_f, l_f = oracle.merge_ml(m_f, l_f, *stats[c][r])
        a = oracle.merge_ml(*stats[0][r], *stats[1][r])
        b = oracle.merge_ml(*stats[2][r], *stats[3][r])
        m_t, l_t = oracle.merge_ml(*oracle.merge_ml(*a, *b), *stats[4][r])
        assert not math.isnan(l_f) and not math.isnan(l_t)
        assert m_t == m_f
        assert abs(l_t - l_f) <= 1e-12 * max(1.0, l_f)
        lse_f = m_f + math.log(l_f) if l_f > 0 else NEG_INF
        if r == g["fully_masked_row"]:
            assert l_f == 0.0 and m_f == NEG_INF and lse_f == NEG_INF
            assert ref[r] == NEG_INF and lse_def[r] == NEG_INF
        else:
            assert abs(lse_f - ref[r]) < 1e-12
            assert abs(lse_def[r] - ref[r]) < 1e-12


def test_lesson_merge_on_lse_partials():
    """The same chunks merged as (lse_c) partials by the oracle's merge (d = 0)."""
    X = si.lesson_matrix(seed=3).double().numpy()
    parts = np.stack([oracle.softmax_rows(c)[1] for c in _lesson_chunks(X)])
    _, lse = oracle.lse_merge(None, parts)
    ref = torch.logsumexp(torch.from_numpy(X), -1).numpy()
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref))
    fin = np.isfinite(ref)
    np.testing.assert_allclose(lse[fin], ref[fin], rtol=0, atol=1e-12)
    # merge order does not matter
    _, lse_rev = oracle.lse_merge(None, parts[::-1].copy())
    np.testing.assert_allclose(lse_rev[fin], lse[fin], rtol=0, atol=1e-13)


def test_naive_merge_is_nan_and_oracle_merge_is_not():
    """Interview lesson: the naive merge gives NaN when both sides are -inf."""
    m_bad = NEG_INF
    with np.errstate(invalid="ignore"):
        naive_l = 0.0 * np.exp(np.float64(m_bad) - max(m_bad, m_bad))
    assert math.isnan(naive_l)
    m, l = oracle.merge_ml(NEG_INF, 0.0, NEG_INF, 0.0)
    assert m == NEG_INF and l == 0.0
    m, l = oracle.merge_ml(NEG_INF, 0.0, 2.0, 3.0)  # one empty side has no weight
    assert m == 2.0 and l == 3.0


# ---------------------------------------------------------------------------
# Row softmax: library routines, closed forms, special cases
# ---------------------------------------------------------------------------

def test_softmax_rows_vs_torch_fp64():
    x, full, pre, _ = si.softmax_input(64, 301, seed=5, frac_full=0.05, frac_prefix=0.2)
    xd = x.double()
    y, lse = oracle.softmax_rows(x.numpy())
    ref_lse = torch.logsumexp(xd, -1).numpy()
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-12)
    ref_y = torch.softmax(xd[torch.from_numpy(fin)], -1).numpy()
    np.testing.assert_allclose(y[fin], ref_y, rtol=1e-12, atol=1e-300)
    # fully -inf rows: +0.0 everywhere, no NaN
    assert np.all(y[~fin] == 0.0) and not np.any(np.signbit(y[~fin]))
    assert len(full) > 0 and np.all(~fin[full.numpy()])
    # -inf elements get exactly +0.0
    assert np.all(y[np.isneginf(x.numpy())] == 0.0)


def test_softmax_closed_forms():
    n = 37
    c = 2.75
    y, lse = oracle.softmax_rows(np.full((1, n), c))
    np.testing.assert_allclose(y[0], 1.0 / n, rtol=1e-15)
    assert abs(lse[0] - (c + math.log(n))) < 1e-14
    # sum to one, and invariance to a constant shift
    x = np.random.default_rng(1).normal(size=(4, 100)) * 5
    y, lse = oracle.softmax_rows(x)
    np.testing.assert_allclose(y.sum(1), 1.0, rtol=1e-14)
    y2, lse2 = oracle.softmax_rows(x + 123.0)
    np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(lse2, lse + 123.0, rtol=1e-15)
    # two-element closed form
    y, lse = oracle.softmax_rows(np.array([[0.0, math.log(3.0)]]))
    np.testing.assert_allclose(y[0], [0.25, 0.75], rtol=1e-15)


def test_softmax_fp32_overflow_argument():
    """Page 'Online softmax in attention': fp32 exp(89) overflows; the safe form does not."""
    g = golden("fp32_exp_overflow.json")
    a = g["overflowing_argument"]
    with np.errstate(over="ignore"):
        assert np.isinf(np.exp(np.float32(a)))
    y, lse = oracle.softmax_rows(np.array([[a, 0.0]], dtype=np.float32))
    assert np.all(np.isfinite(y)) and np.isfinite(lse[0])
    e = math.exp(-a)
    np.testing.assert_allclose(y[0], [1.0 / (1.0 + e), e / (1.0 + e)], rtol=1e-15)


def test_softmax_dtype_widening_is_exact():
    x = si.randn((3, 50), seed=9, dtype=torch.bfloat16, mul=3.0)
    y16, l16 = oracle.softmax_rows(bf16_bits(x))
    y64, l64 = oracle.softmax_rows(x.double().numpy())
    np.testing.assert_array_equal(y16, y64)
    np.testing.assert_array_equal(l16, l64)


# ---------------------------------------------------------------------------
# Attention: SDPA in fp64, closed forms, invariants, brute force (FA-1 order)
# ---------------------------------------------------------------------------

def _lower_right_mask(Nq, Nk):
    """torch's own lower-right causal mask (query i sees key j iff j <= i + Nk - Nq): an
    independent statement of the bottom-right reading the oracle implements."""
    import warnings

    from torch.nn.attention.bias import causal_lower_right

    with warnings.catch_warnings():
        warnings.simplefilter("ignore")  # torch warns that Nq > Nk leaves rows without keys
        return causal_lower_right(Nq, Nk)._materialize(torch.device("cpu"))


def _sdpa_ref(q, k, v, causal, scale, kv_len=None):
    """fp64 library reference with an explicit boolean mask, plus logsumexp of the scores.  Rows with
    no visible key (SDPA gives NaN there) are returned as O = 0, their logsumexp is -inf."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    vis = torch.ones(B, 1, Nq, Nk, dtype=torch.bool)
    if causal:
        vis &= _lower_right_mask(Nq, Nk)
    if kv_len is not None:
        vis &= (torch.arange(Nk)[None, :] < torch.as_tensor(kv_len)[:, None]).view(B, 1, 1, Nk)
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=vis, scale=scale)
    o = torch.where(vis.any(-1, keepdim=True), o, torch.zeros_like(o))
    s = torch.einsum("bhid,bhjd->bhij", q, k) * scale
    s = s.masked_fill(~vis, NEG_INF)
    return o, torch.logsumexp(s, -1), vis


@pytest.mark.parametrize("N,Nk,d", golden("lesson_step2_shapes.json")["cases"])
def test_attention_vs_sdpa_lesson_shapes(N, Nk, d):
    q, k, v = si.attn_inputs(1, 1, N, Nk, d, torch.float64, seed=N * 100 + Nk)
    o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    ro, rl, _ = _sdpa_ref(q, k, v, False, 1 / math.sqrt(d))
    np.testing.assert_allclose(o, ro.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_vs_sdpa_masked(causal):
    B, H, N, d = 3, 2, 37, 16
    q, k, v = si.attn_inputs(B, H, N, N, d, torch.float64, seed=11)
    kv_len = [37, 1, 20]
    o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), causal=causal, kv_len=kv_len)
    ro, rl, _ = _sdpa_ref(q, k, v, causal, 1 / math.sqrt(d), kv_len)
    np.testing.assert_allclose(o, ro.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("Nq,Nk", [(1, 9), (3, 11), (7, 7), (5, 40), (12, 5), (4, 1)])
def test_attention_kv_cache_causal_vs_lower_right_sdpa(Nq, Nk):
    # Nq new queries against Nk keys (chunked prefill / multi-token decode): the queries are the last
    # Nq positions, so query i sees keys j <= i + Nk - Nq -- torch's lower-right causal mask.  With
    # Nq > Nk the first Nq - Nk queries see no key: O = +0.0 and LSE = -inf, no NaN.
    B, H, d = 2, 3, 8
    q, k, v = si.attn_inputs(B, H, Nq, Nk, d, torch.float64, seed=40 + Nq * 7 + Nk)
    o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), causal=True)
    ro, rl, vis = _sdpa_ref(q, k, v, True, 1 / math.sqrt(d))
    assert not np.isnan(o).any() and not np.isnan(lse).any()
    np.testing.assert_allclose(o, ro.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(rl.numpy()))
    fin = np.isfinite(rl.numpy())
    np.testing.assert_allclose(lse[fin], rl.numpy()[fin], rtol=0, atol=1e-12)
    empty = ~vis.any(-1).expand(B, H, Nq).numpy()
    assert empty.sum() == B * H * max(0, Nq - Nk)
    assert np.all(o[empty] == 0.0) and not np.any(np.signbit(o[empty]))


def test_attention_kv_cache_causal_closed_forms():
    # K == 0: every visible score is 0, so query i averages V_0 .. V_{i + Nk - Nq} and LSE = ln(i + Nk - Nq + 1)
    Nq, Nk, d = 4, 10, 3
    rng = np.random.default_rng(8)
    q, v = rng.standard_normal((1, 1, Nq, d)), rng.standard_normal((1, 1, Nk, d))
    o, lse = oracle.attention(q, np.zeros((1, 1, Nk, d)), v, causal=True)
    for i in range(Nq):
        last = i + Nk - Nq
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :last + 1].mean(0), rtol=1e-13, atol=1e-14)
        assert lse[0, 0, i] == pytest.approx(math.log(last + 1), abs=1e-14)
    # one new query sees the whole cache: causal is the same as non-causal
    q1 = rng.standard_normal((2, 2, 1, d))
    k1, v1 = rng.standard_normal((2, 2, 17, d)), rng.standard_normal((2, 2, 17, d))
    oc, lc = oracle.attention(q1, k1, v1, causal=True)
    on, ln_ = oracle.attention(q1, k1, v1, causal=False)
    np.testing.assert_array_equal(oc, on)
    np.testing.assert_array_equal(lc, ln_)


def test_attention_chunked_prefill_equals_last_rows_of_full_causal():
    # the last Nq rows of causal attention over a whole sequence of N tokens are the causal attention
    # of those Nq queries against all N keys (the chunk after a cache of N - Nq keys)
    N, Nq, d = 23, 6, 8
    q, k, v = si.attn_inputs(2, 2, N, N, d, torch.float64, seed=44)
    of, lf = oracle.attention(q.numpy(), k.numpy(), v.numpy(), causal=True)
    oc, lc = oracle.attention(q[:, :, N - Nq:].contiguous().numpy(), k.numpy(), v.numpy(), causal=True)
    np.testing.assert_array_equal(oc, of[:, :, N - Nq:])
    np.testing.assert_array_equal(lc, lf[:, :, N - Nq:])


def test_attention_scale_and_noncausal_rectangular():
    B, H, Nq, Nk, d = 2, 3, 5, 29, 8
    q, k, v = si.attn_inputs(B, H, Nq, Nk, d, torch.float64, seed=12)
    for scale in (0.1, 1.0, 2.5):
        o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), scale=scale)
        ro, rl, _ = _sdpa_ref(q, k, v, False, scale)
        np.testing.assert_allclose(o, ro.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, rl.numpy(), rtol=0, atol=1e-12)


def test_attention_closed_forms():
    B, H, N, d = 2, 2, 19, 8
    q, k, v = si.attn_inputs(B, H, N, N, d, torch.float64, seed=13)
    qn, kn, vn = q.numpy(), k.numpy(), v.numpy()
    scale = 1 / math.sqrt(d)
    # causal row 0 sees only key 0: O_0 = V_0, LSE_0 = scale * q_0 . k_0
    o, lse = oracle.attention(qn, kn, vn, causal=True)
    np.testing.assert_array_equal(o[:, :, 0], vn[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], scale * np.einsum("bhd,bhd->bh", qn[:, :, 0], kn[:, :, 0]),
                               rtol=0, atol=1e-14)
    # kv_len = 1: every row sees only key 0
    o, lse = oracle.attention(qn, kn, vn, kv_len=[1, 1])
    np.testing.assert_array_equal(o, np.broadcast_to(vn[:, :, :1], o.shape))
    # K == 0: uniform weights over the visible keys
    kz = np.zeros_like(kn)
    o, lse = oracle.attention(qn, kz, vn, kv_len=[N, 7])
    np.testing.assert_allclose(o[0], np.broadcast_to(vn[0].mean(1, keepdims=True), o[0].shape), atol=1e-14)
    np.testing.assert_allclose(o[1], np.broadcast_to(vn[1, :, :7].mean(1, keepdims=True), o[1].shape), atol=1e-14)
    np.testing.assert_allclose(lse[0], math.log(N), atol=1e-14)
    np.testing.assert_allclose(lse[1], math.log(7), atol=1e-14)
    # causal + K == 0: row i averages V_0..V_i, LSE = ln(i + 1)
    o, lse = oracle.attention(qn, kz, vn, causal=True)
    csum = np.cumsum(vn, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    np.testing.assert_allclose(o, csum, atol=1e-14)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, N + 1)), lse.shape), atol=1e-14)
    # no visible key: O = +0.0, LSE = -inf, no NaN
    o, lse = oracle.attention(qn, kn, vn, kv_len=[0, N])
    assert np.all(o[0] == 0.0) and not np.any(np.signbit(o[0])) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(o[1]))


def test_attention_permutation_invariance():
    B, H, Nq, Nk, d = 1, 2, 9, 23, 8
    q, k, v = si.attn_inputs(B, H, Nq, Nk, d, torch.float64, seed=14)
    perm = torch.randperm(Nk, generator=torch.Generator().manual_seed(2))
    o1, l1 = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    o2, l2 = oracle.attention(q.numpy(), k[:, :, perm].numpy(), v[:, :, perm].numpy())
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-13)


def test_attention_rows_subset_and_bf16_widening():
    B, H, N, d = 2, 3, 40, 16
    q, k, v = si.attn_inputs(B, H, N, N, d, torch.bfloat16, seed=15)
    of, lf = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True)
    o64, l64 = oracle.attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), causal=True)
    np.testing.assert_array_equal(of, o64)
    np.testing.assert_array_equal(lf, l64)
    rows = np.array([0, 5, 39, 40, 119, 200, 239])
    o_s, l_s = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True, rows=rows)
    np.testing.assert_array_equal(o_s, of.reshape(-1, d)[rows])
    np.testing.assert_array_equal(l_s, lf.reshape(-1)[rows])


def test_fa1_block_order_reaches_definition():
    """Brute force of the lesson's V1 loop (Br=4, Bc=3) against the materialised
    definition: the online block merge is exact up to rounding."""
    ws = golden("lesson_step2_shapes.json")["walk_shapes"]
    q, k, v = si.attn_inputs(1, 1, ws["N"], ws["Nk"], ws["d"], torch.float32, seed=0)
    qd, kd, vd = (t[0, 0].double().numpy() for t in (q, k, v))
    o_fa1 = oracle.attention_fa1(qd, kd, vd, Br=ws["Br"], Bc=ws["Bc"])
    o_def, _ = oracle.attention(qd[None, None], kd[None, None], vd[None, None])
    np.testing.assert_allclose(o_fa1, o_def[0, 0], rtol=0, atol=1e-12)
    for N, Nk, d in golden("lesson_step2_shapes.json")["cases"]:
        q, k, v = si.attn_inputs(1, 1, N, Nk, d, torch.float64, seed=7 + N)
        for Br, Bc in ((4, 3), (1, 1), (3, 5), (64, 64)):
            o_fa1 = oracle.attention_fa1(q[0, 0].numpy(), k[0, 0].numpy(), v[0, 0].numpy(), Br=Br, Bc=Bc)
            o_def, _ = oracle.attention(q.numpy(), k.numpy(), v.numpy())
            np.testing.assert_allclose(o_fa1, o_def[0, 0], rtol=0, atol=1e-12)


def test_lesson_fa1_page_tolerance_against_sdpa():
    """The lesson's own check, atol 1e-5, on the same shapes (float32 inputs as on the page)."""
    g = golden("lesson_step2_shapes.json")
    for N, Nk, d in g["cases"]:
        q, k, v = si.attn_inputs(1, 1, N, Nk, d, torch.float32, seed=N)
        o = oracle.attention_fa1(q[0, 0].double().numpy(), k[0, 0].double().numpy(), v[0, 0].double().numpy())
        ref = F.scaled_dot_product_attention(q[0], k[0], v[0])[0].double().numpy()
        assert np.max(np.abs(o - ref)) < g["atol"]


# ---------------------------------------------------------------------------
# Split-KV partials and their merge
# ---------------------------------------------------------------------------

def _partials(q, k, v, chunk, kv_len=None):
    """Per-chunk oracle attention over key slices; chunks beyond kv_len are empty."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    S = (Nk + chunk - 1) // chunk
    po = np.zeros((S, B * H * Nq, d))
    pl = np.zeros((S, B * H * Nq))
    for c in range(S):
        j0, j1 = c * chunk, min(Nk, (c + 1) * chunk)
        kl = None
        if kv_len is not None:
            kl = np.clip(np.asarray(kv_len) - j0, 0, j1 - j0)
        o, l = oracle.attention(q, k[:, :, j0:j1], v[:, :, j0:j1], kv_len=kl)
        po[c] = o.reshape(-1, d)
        pl[c] = l.reshape(-1)
    return po, pl


def _brute_attention_rows(q, k, v, causal, scale):
    """softmax(q k^T scale) v for one head in plain fp64 numpy, -inf where masked (causal: key j
    hidden from query i when j > i + Nk - Nq, the queries being the sequence's last Nq positions)."""
    s = (q @ k.T) * scale
    if causal:
        off = k.shape[0] - q.shape[0]
        s = np.where(np.arange(k.shape[0])[None, :] > np.arange(q.shape[0])[:, None] + off, -np.inf, s)
    m = s.max(axis=1, keepdims=True) if s.shape[1] else np.full((s.shape[0], 1), -np.inf)
    o = np.zeros((q.shape[0], v.shape[1]))
    lse = np.full(q.shape[0], -np.inf)
    for i in range(q.shape[0]):
        if not np.isfinite(m[i, 0]):
            continue
        w = np.exp(s[i] - m[i, 0])
        o[i] = (w @ v) / w.sum()
        lse[i] = m[i, 0] + np.log(w.sum())
    return o, lse


def test_attention_grouped_heads_reduce_to_repeated_heads():
    # grouped key/value heads: query head h reads head h // (H // Hkv).  Pinned to the per-head
    # oracle with K and V repeated across each group, and to brute force for one head.
    rng = np.random.default_rng(5)
    B, H, Hkv, Nq, Nk, d = 2, 6, 2, 7, 9, 8
    q = rng.standard_normal((B, H, Nq, d))
    k = rng.standard_normal((B, Hkv, Nk, d))
    v = rng.standard_normal((B, Hkv, Nk, d))
    for causal in (False, True):
        og, lg = oracle.attention(q, k, v, causal=causal, kv_len=[9, 4])
        orp, lrp = oracle.attention(q, np.repeat(k, H // Hkv, axis=1), np.repeat(v, H // Hkv, axis=1),
                                    causal=causal, kv_len=[9, 4])
        np.testing.assert_array_equal(og, orp)
        np.testing.assert_array_equal(lg, lrp)
    # brute force: batch 1, query head 5 uses key/value head 1 over the first 4 keys
    ob, lb = _brute_attention_rows(q[1, 5], k[1, 1, :4], v[1, 1, :4], False, 1 / math.sqrt(d))
    og, lg = oracle.attention(q, k, v, kv_len=[9, 4])
    np.testing.assert_allclose(og[1, 5], ob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lg[1, 5], lb, rtol=1e-12, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.attention(q, k[:, :1].repeat(4, axis=1), v[:, :1].repeat(4, axis=1))  # 4 does not divide 6


def test_attention_varlen_equal_lengths_is_dense_batch():
    # packed token-major sequences of one length N equal the dense [B, H, N, d] batch
    rng = np.random.default_rng(6)
    B, H, Hkv, N, d = 3, 4, 2, 10, 8
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    pack = lambda t: np.ascontiguousarray(t.transpose(0, 2, 1, 3).reshape(B * N, t.shape[1], d))
    cu = np.arange(0, (B + 1) * N, N)
    for causal in (False, True):
        od, ld = oracle.attention(q, k, v, causal=causal)
        ov, lv = oracle.attention_varlen(pack(q), pack(k), pack(v), cu, cu, causal=causal)
        np.testing.assert_array_equal(ov, pack(od))
        np.testing.assert_array_equal(lv, ld.transpose(0, 2, 1).reshape(B * N, H))


def test_attention_varlen_brute_force_mixed_lengths():
    # mixed lengths, a sequence without keys (O = 0, lse = -inf), one without queries, and causal
    # with more keys than queries (key j visible to query i iff j <= i + lk - lq within the sequence)
    rng = np.random.default_rng(7)
    H, Hkv, d = 4, 2, 8
    lq, lk = [5, 3, 0, 6], [7, 0, 2, 6]
    cq, ck = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    q = rng.standard_normal((cq[-1], H, d))
    k = rng.standard_normal((ck[-1], Hkv, d))
    v = rng.standard_normal((ck[-1], Hkv, d))
    sc = 0.3
    for causal in (False, True):
        ov, lv = oracle.attention_varlen(q, k, v, cq, ck, causal=causal, scale=sc)
        for s in range(len(lq)):
            for h in range(H):
                ob, lb = _brute_attention_rows(q[cq[s]:cq[s + 1], h], k[ck[s]:ck[s + 1], h // 2],
                                               v[ck[s]:ck[s + 1], h // 2], causal, sc)
                np.testing.assert_allclose(ov[cq[s]:cq[s + 1], h], ob, rtol=1e-12, atol=1e-12)
                np.testing.assert_array_equal(np.isneginf(lv[cq[s]:cq[s + 1], h]), np.isneginf(lb))
                fin = np.isfinite(lb)
                np.testing.assert_allclose(lv[cq[s]:cq[s + 1], h][fin], lb[fin], rtol=1e-12, atol=1e-12)
    assert np.all(ov[cq[1]:cq[2]] == 0) and np.all(np.isneginf(lv[cq[1]:cq[2]]))


def _autograd_bwd(q, k, v, dout, causal, scale):
    """fp64 torch autograd of softmax(scale Q K^T, masked) V: the library's derivative."""
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:
        Nq, Nk = s.shape[-2:]
        s = s.masked_fill(~_lower_right_mask(Nq, Nk), float("-inf"))
    # a row without a visible key (Nq > Nk) has a constant zero output, so no gradient
    p = torch.nan_to_num(torch.softmax(s, dim=-1), nan=0.0)
    o = p @ tv
    o.backward(torch.tensor(dout, dtype=torch.float64))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(7, 7), (5, 9), (9, 5)])
def test_attention_bwd_vs_fp64_autograd(causal, Nq, Nk):
    rng = np.random.default_rng(Nq * 10 + Nk)
    q = rng.standard_normal((2, 3, Nq, 8))
    k = rng.standard_normal((2, 3, Nk, 8))
    v = rng.standard_normal((2, 3, Nk, 8))
    do = rng.standard_normal((2, 3, Nq, 8))
    got = oracle.attention_bwd(q, k, v, do, causal=causal, scale=0.4)
    ref = _autograd_bwd(q, k, v, do, causal, 0.4)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_bwd_grouped_heads_vs_fp64_autograd(causal):
    # key/value heads shared by groups of query heads: torch's autograd through K, V repeated over each
    # group sums the gradient of every use, which is the definition the oracle must reach
    rng = np.random.default_rng(31 + causal)
    B, H, Hkv, N, d = 2, 6, 2, 7, 5
    q, do = rng.standard_normal((B, H, N, d)), rng.standard_normal((B, H, N, d))
    k, v = rng.standard_normal((B, Hkv, N, d)), rng.standard_normal((B, Hkv, N, d))
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    g = H // Hkv
    s = 0.3 * tq @ tk.repeat_interleave(g, dim=1).transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.arange(N)[None, :] > torch.arange(N)[:, None], float("-inf"))
    (torch.softmax(s, dim=-1) @ tv.repeat_interleave(g, dim=1)).backward(torch.tensor(do))
    got = oracle.attention_bwd(q, k, v, do, causal=causal, scale=0.3)
    for a, r in zip(got, (tq.grad, tk.grad, tv.grad)):
        np.testing.assert_allclose(a, r.numpy(), rtol=1e-11, atol=1e-12)
    # with H_kv = H it is the ungrouped backward of each head
    full = oracle.attention_bwd(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), do, causal=causal, scale=0.3)
    np.testing.assert_allclose(got[0], full[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(got[1], full[1].reshape(B, Hkv, g, N, d).sum(2), rtol=1e-11, atol=1e-12)


def test_attention_bwd_varlen_vs_fp64_autograd():
    # packed sequences of mixed lengths (one without keys, one without queries, causal with more keys than
    # queries): every token's gradient is that of its own sequence, computed here by torch autograd
    lq, lk = [5, 0, 7, 3, 6, 4], [5, 4, 7, 0, 9, 2]
    H, Hkv, d = 4, 2, 6
    rng = np.random.default_rng(77)
    Tq, Tk = sum(lq), sum(lk)
    q, do = rng.standard_normal((Tq, H, d)), rng.standard_normal((Tq, H, d))
    k, v = rng.standard_normal((Tk, Hkv, d)), rng.standard_normal((Tk, Hkv, d))
    cq, ck = np.cumsum([0] + lq), np.cumsum([0] + lk)
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd_varlen(q, k, v, do, cq, ck, causal=causal, scale=0.4)
        rq, rk, rv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for s in range(len(lq)):
            if lq[s] == 0 or lk[s] == 0:
                continue
            sl_q, sl_k = slice(cq[s], cq[s + 1]), slice(ck[s], ck[s + 1])
            tq, tk, tv = (torch.tensor(a.transpose(1, 0, 2), requires_grad=True) for a in (q[sl_q], k[sl_k], v[sl_k]))
            sc = 0.4 * tq @ tk.repeat_interleave(H // Hkv, 0).transpose(-1, -2)
            if causal:
                sc = sc.masked_fill(~_lower_right_mask(lq[s], lk[s]), float("-inf"))
            out = torch.nan_to_num(torch.softmax(sc, -1), nan=0.0) @ tv.repeat_interleave(H // Hkv, 0)
            out.backward(torch.tensor(do[sl_q].transpose(1, 0, 2)))
            rq[sl_q], rk[sl_k], rv[sl_k] = (t.grad.numpy().transpose(1, 0, 2) for t in (tq, tk, tv))
        for a, r in ((dq, rq), (dk, rk), (dv, rv)):
            np.testing.assert_allclose(a, r, rtol=1e-11, atol=1e-12)
        # the key-less sequence's queries and the query-less sequence's keys get exactly zero
        assert np.all(dq[cq[3]:cq[4]] == 0.0) and np.all(dk[ck[1]:ck[2]] == 0.0) and np.all(dv[ck[1]:ck[2]] == 0.0)


def test_attention_bwd_finite_differences():
    # central differences of L = sum(O * dO) through the (pinned) forward oracle
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((1, 1, n, 3)) for n in (4, 5, 5))
    do = rng.standard_normal((1, 1, 4, 3))
    for causal in (False, True):
        grads = oracle.attention_bwd(q, k, v, do, causal=causal, scale=0.7)

        def loss(qq, kk, vv):
            o, _ = oracle.attention(qq, kk, vv, causal=causal, scale=0.7)
            return float(np.sum(o * do))

        h = 1e-6
        for which, (arr, g) in enumerate(zip((q, k, v), grads)):
            for idx in np.ndindex(arr.shape):
                a = [q.copy(), k.copy(), v.copy()]
                a[which][idx] += h
                up = loss(*a)
                a[which][idx] -= 2 * h
                dn = loss(*a)
                assert abs((up - dn) / (2 * h) - g[idx]) < 1e-6, (which, idx)


def test_attention_bwd_closed_forms():
    rng = np.random.default_rng(4)
    q, k, v = (rng.standard_normal((1, 2, 6, 4)) for _ in range(3))
    do = rng.standard_normal((1, 2, 6, 4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do)
    # every row's weights sum to 1, so the value gradients sum to the output gradients
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), rtol=1e-12, atol=1e-12)
    # causal with one query per visible key at row 0: a single visible key has weight 1 whatever
    # the scores, so row 0 of dQ is zero
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=True)
    np.testing.assert_array_equal(dq[:, :, 0], 0.0)
    # the last key is seen only by the last query: dV[last] = P[last, last] dO[last]
    s5 = np.einsum("bhe,bhje->bhj", q[:, :, 5], k) / math.sqrt(4)
    p55 = np.exp(s5[..., 5] - s5.max(-1)) / np.exp(s5 - s5.max(-1, keepdims=True)).sum(-1)
    np.testing.assert_allclose(dv[:, :, 5], p55[..., None] * do[:, :, 5], rtol=1e-12)
    # a single key overall: no score gradient at all
    dq, dk, dv = oracle.attention_bwd(q, k[:, :, :1], v[:, :, :1], do)
    np.testing.assert_array_equal(dq, 0.0)
    np.testing.assert_array_equal(dk, 0.0)
    np.testing.assert_allclose(dv[:, :, 0], do.sum(axis=2), rtol=1e-12)


@pytest.mark.parametrize("causal,Nq,Nk", [(False, 9, 13), (True, 11, 11), (False, 1, 1), (True, 6, 14), (True, 9, 4)])
def test_attention_bwd_sampled_vs_fp64_autograd(causal, Nq, Nk):
    # the row-sampled gradients against torch's fp64 autograd, at every row and at a shuffled subset
    rng = np.random.default_rng(100 + Nq)
    q, k, v = rng.standard_normal((Nq, 6)), rng.standard_normal((Nk, 6)), rng.standard_normal((Nk, 6))
    do = rng.standard_normal((Nq, 6))
    rq, rk, rv = _autograd_bwd(q, k, v, do, causal, 0.5)
    dq, dk, dv = oracle.attention_bwd_sampled(q, k, v, do, np.arange(Nq), np.arange(Nk), causal=causal, scale=0.5)
    for g, r in ((dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(g, r, rtol=1e-11, atol=1e-12)
    qi, kj = rng.permutation(Nq)[: max(1, Nq // 2)], rng.permutation(Nk)[: max(1, Nk // 3)]
    dq, dk, dv = oracle.attention_bwd_sampled(q, k, v, do, qi, kj, causal=causal, scale=0.5)
    np.testing.assert_allclose(dq, rq[qi], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, rk[kj], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, rv[kj], rtol=1e-11, atol=1e-12)


def test_attention_bwd_sampled_bf16_matches_full():
    # bf16 bit patterns widen exactly on both paths, so the sampled rows equal the full gradients
    q, k, v = si.attn_inputs(1, 1, 40, 40, 16, torch.bfloat16, seed=21)
    do = si.randn((1, 1, 40, 16), 24, torch.bfloat16)
    full = oracle.attention_bwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), bf16_bits(do), causal=True)
    rows = np.array([0, 17, 39])
    got = oracle.attention_bwd_sampled(bf16_bits(q[0, 0]), bf16_bits(k[0, 0]), bf16_bits(v[0, 0]),
                                       bf16_bits(do[0, 0]), rows, rows, causal=True)
    for g, f in zip(got, full):
        np.testing.assert_allclose(g, f[0, 0][rows], rtol=1e-12, atol=1e-13)


def test_lse_merge_reaches_unsplit_attention():
    B, H, Nq, Nk, d = 3, 2, 2, 50, 8
    q, k, v = si.attn_inputs(B, H, Nq, Nk, d, torch.float64, seed=16)
    qn, kn, vn = q.numpy(), k.numpy(), v.numpy()
    kv_len = [50, 9, 0]
    po, pl = _partials(qn, kn, vn, 7, kv_len)
    o, lse = oracle.lse_merge(po, pl)
    ro, rl = oracle.attention(qn, kn, vn, kv_len=kv_len)
    np.testing.assert_allclose(o, ro.reshape(-1, d), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(rl.reshape(-1)))
    fin = np.isfinite(rl.reshape(-1))
    np.testing.assert_allclose(lse[fin], rl.reshape(-1)[fin], rtol=0, atol=1e-12)
    # batch 2 has no key at all: O = +0.0, LSE = -inf
    last = slice(2 * H * Nq, 3 * H * Nq)
    assert np.all(o[last] == 0.0) and np.all(np.isneginf(lse[last]))
    # the merge is order-free
    perm = np.random.default_rng(0).permutation(po.shape[0])
    o2, l2 = oracle.lse_merge(po[perm], pl[perm])
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)


def test_lse_merge_closed_forms():
    # two equal partials: same o, lse + ln 2
    po = np.array([[[1.0, -2.0]], [[1.0, -2.0]]])
    pl = np.array([[0.5], [0.5]])
    o, lse = oracle.lse_merge(po, pl)
    np.testing.assert_allclose(o[0], [1.0, -2.0], rtol=1e-15)
    assert abs(lse[0] - (0.5 + math.log(2.0))) < 1e-15
    # weights e^a/(e^a+e^b)
    po = np.array([[[2.0]], [[-4.0]]])
    pl = np.array([[1.0], [3.0]])
    o, lse = oracle.lse_merge(po, pl)
    w = 1.0 / (1.0 + math.exp(2.0))
    assert abs(o[0, 0] - (2.0 * w - 4.0 * (1 - w))) < 1e-14
    # an empty partial (-inf, o = 0) has no weight; all empty gives 0 and -inf
    po = np.array([[[5.0]], [[0.0]]])
    pl = np.array([[0.25], [NEG_INF]])
    o, lse = oracle.lse_merge(po, pl)
    assert o[0, 0] == 5.0 and lse[0] == 0.25
    o, lse = oracle.lse_merge(np.zeros((3, 1, 2)), np.full((3, 1), NEG_INF))
    assert np.all(o == 0.0) and np.isneginf(lse[0])


def test_synth_recipes():
    x, full, pre, lens = si.softmax_input(4096, 64, seed=0)
    assert len(full) == 41 and len(pre) == 410
    assert set(full.tolist()).isdisjoint(pre.tolist())
    xn = x.numpy()
    assert np.all(np.isneginf(xn[full.numpy()]))
    for r, n in zip(pre.tolist()[:20], lens.tolist()[:20]):
        assert np.all(np.isneginf(xn[r, :n])) and np.all(np.isfinite(xn[r, n:]))
    kv = si.decode_kv_len(32, 32768, seed=0)
    assert kv.dtype == torch.int32 and int((kv < 32768).sum()) <= 2 and int(kv.min()) >= 1
    r = si.sample_rows(1000, 40, seed=0)
    assert r[0] == 0 and r[-1] == 999 and 127 in r.tolist() and 128 in r.tolist()
