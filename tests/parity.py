"""Comparison helpers for the GPU parity tests (GPU output vs the fp64 oracle).

Tolerances (stated by the workload definitions, applied element by element):
  bf16 attention output O        max |O - O_ref|          <= 2e-2
  fp32 row softmax y             |y - y_ref| <= 1e-5 |y_ref|, and y_ref == 0 -> y is exactly +0.0
  LSE (every kernel)             |lse - lse_ref|           <= 1e-4, -inf exactly where the reference is -inf
  fp32 attention (tiny worked)   max |O - O_ref|          <= 1e-5
No output may be NaN.  Rows with no visible key must be exactly +0.0 with LSE -inf.
"""
import numpy as np
import torch

BF16_O_ATOL = 2e-2
SOFTMAX_RTOL = 1e-5
LSE_ATOL = 1e-4
F32_ATTN_ATOL = 1e-5


def to_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (what the oracle widens exactly)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_no_nan(a, what):
    a = to_np(a)
    assert not np.isnan(a).any(), f"{what}: NaN in output"


def assert_softmax_close(y, y_ref, rtol=SOFTMAX_RTOL, what="y"):
    y, r = to_np(y), np.asarray(y_ref, np.float64)
    assert y.shape == r.shape
    assert_no_nan(y, what)
    zero = r == 0.0
    assert np.all(y[zero] == 0.0), f"{what}: expected exact zeros"
    assert not np.any(np.signbit(y[zero])), f"{what}: expected +0.0"
    err = np.abs(y - r)
    bad = err > rtol * np.abs(r)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / np.maximum(np.abs(r), 1e-300), 0)), r.shape)
        raise AssertionError(f"{what}: {bad.sum()} elements beyond rel {rtol}; worst at {i}: {y[i]!r} vs {r[i]!r}")


def assert_lse_close(lse, lse_ref, atol=LSE_ATOL, what="lse"):
    a, r = to_np(lse).reshape(-1), np.asarray(lse_ref, np.float64).reshape(-1)
    assert a.shape == r.shape
    assert_no_nan(a, what)
    ninf = np.isneginf(r)
    assert np.array_equal(np.isneginf(a), ninf), f"{what}: -inf pattern differs"
    fin = ~ninf
    if fin.any():
        err = np.abs(a[fin] - r[fin])
        assert err.max() <= atol, f"{what}: max abs err {err.max():.3e} > {atol} at {np.argmax(err)}"


def assert_out_close(o, o_ref, atol, lse_ref=None, what="O"):
    a, r = to_np(o), np.asarray(o_ref, np.float64)
    assert a.shape == r.shape, (a.shape, r.shape)
    assert_no_nan(a, what)
    err = np.abs(a - r)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= atol, f"{what}: max abs err {err.max():.3e} > {atol} at {worst}"
    if lse_ref is not None:
        empty = np.isneginf(np.asarray(lse_ref).reshape(-1))
        if empty.any():
            rows = a.reshape(empty.shape[0], -1)[empty]
            assert np.all(rows == 0.0) and not np.any(np.signbit(rows)), f"{what}: empty rows must be +0.0"
    return float(err.max())
