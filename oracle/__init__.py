"""CPU oracle for online-softmax attention: test infrastructure, not product.

This package is the plain, slow, obviously-correct fp64 definition of what the
GPU library computes.  It shares no code with the CUDA path and neither
imports the other.  Only the test-suite, the smoke check and the bench's
CPU-baseline leg may import it; the product path never does.

The arithmetic lives in ``oracle.c`` (plain C11, fp64, one thread pool over
independent rows).  This module only marshals numpy arrays to it and builds
the shared object with gcc on first use.

Pins: every function here is checked in ``tests/test_oracle.py`` against the
pages' printed worked examples (``tests/golden/``), closed forms, invariants,
brute force and fp64 library routines.  None is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboa_oracle.so")
_lock = threading.Lock()
_lib = None

F64, F32, BF16 = 0, 1, 2

_c_dbl_p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboa_oracle.so next to it (if stale) and return its path."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
                   "-pthread", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_softmax_rows.argtypes = [vp, i32, i64, i64, i64, vp, i64, vp, i32]
    lib.oracle_softmax_rows.restype = i32
    lib.oracle_attn.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i64, i64, i32, dbl, vp, vp, i64, vp, vp, i32]
    lib.oracle_attn.restype = i32
    lib.oracle_attn_bwd.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, i64, i64, i32, dbl, vp, vp, vp, i32]
    lib.oracle_attn_bwd.restype = i32
    lib.oracle_attn_bwd_sampled.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i32, dbl, vp, i64, vp, i64, vp, vp,
                                            vp, i32]
    lib.oracle_attn_bwd_sampled.restype = i32
    lib.oracle_lse_merge.argtypes = [vp, vp, i64, i64, i64, vp, vp]
    lib.oracle_lse_merge.restype = i32
    lib.oracle_online_stats.argtypes = [vp, i64, _c_dbl_p, _c_dbl_p]
    lib.oracle_online_stats.restype = None
    lib.oracle_online_stats_trace.argtypes = [vp, i64, vp, vp]
    lib.oracle_online_stats_trace.restype = None
    lib.oracle_merge_ml.argtypes = [dbl, dbl, dbl, dbl, _c_dbl_p, _c_dbl_p]
    lib.oracle_merge_ml.restype = None
    lib.oracle_attn_fa1.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, dbl, vp]
    lib.oracle_attn_fa1.restype = i32
    _lib = lib
    return lib


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _as_input(a):
    """Return (contiguous array, dtype code).  bf16 arrives as uint16 bit patterns."""
    a = np.asarray(a)
    if a.dtype == np.float64:
        code = F64
    elif a.dtype == np.float32:
        code = F32
    elif a.dtype == np.uint16:
        code = BF16
    else:
        a = a.astype(np.float64)
        code = F64
    return np.ascontiguousarray(a), code


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def softmax_rows(x, nthreads=None):
    """Three-pass safe softmax of each row of a 2-D array, plus its natural log-sum-exp.

    x: [rows, cols] float64/float32, or uint16 holding bf16 bits.  Returns (y, lse) in fp64.
    """
    xa, code = _as_input(x)
    if xa.ndim != 2:
        raise ValueError("x must be 2-D")
    rows, cols = xa.shape
    y = np.empty((rows, cols), np.float64)
    lse = np.empty(rows, np.float64)
    rc = _load().oracle_softmax_rows(_ptr(xa), code, rows, cols, cols, _ptr(y), cols, _ptr(lse), _threads(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_softmax_rows failed")
    return y, lse


def attention(q, k, v, causal=False, scale=None, kv_len=None, rows=None, nthreads=None):
    """Materialised softmax(Q K^T * scale) V and per-row LSE, in fp64.

    q [B,H,Nq,d], k/v [B,Hkv,Nk,d] (same dtype code; Hkv divides H and query head h
    reads key/value head h // (H // Hkv)).  kv_len: None or int array [B] (keys j >= kv_len[b]
    hidden).  causal: the queries are the last Nq positions of the Nk keys' sequence, so key j
    is visible to query i iff j <= i + (Nk - Nq) (j <= i when Nq == Nk).
    rows: None for every row, else flattened row indices (b*H + h)*Nq + i; then the
    result has shape [len(rows), d] and [len(rows)].
    """
    qa, code = _as_input(q)
    ka, kcode = _as_input(k)
    va, vcode = _as_input(v)
    if not (code == kcode == vcode):
        raise ValueError("q, k, v must share a dtype")
    if qa.ndim != 4 or ka.ndim != 4 or va.ndim != 4:
        raise ValueError("q, k, v must be [B,H,N,d]")
    B, H, Nq, d = qa.shape
    Hkv, Nk = ka.shape[1], ka.shape[2]
    if ka.shape != (B, Hkv, Nk, d) or va.shape != (B, Hkv, Nk, d):
        raise ValueError("k/v shape mismatch")
    if Hkv < 1 or H % Hkv != 0:
        raise ValueError("the key/value head count must divide the query head count")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kvl = None
    if kv_len is not None:
        kvl = np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32))
        if kvl.shape != (B,):
            raise ValueError("kv_len must be [B]")
    if rows is None:
        n = B * H * Nq
        ra = None
    else:
        ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = ra.shape[0]
    o = np.zeros((n, d), np.float64)
    lse = np.empty(n, np.float64)
    rc = _load().oracle_attn(_ptr(qa), _ptr(ka), _ptr(va), code, B, H, Hkv, Nq, Nk, d, int(bool(causal)),
                             float(scale), _ptr(kvl), _ptr(ra), n, _ptr(o), _ptr(lse), _threads(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn failed")
    if rows is None:
        return o.reshape(B, H, Nq, d), lse.reshape(B, H, Nq)
    return o, lse


def attention_bwd(q, k, v, dout, causal=False, scale=None, nthreads=None):
    """Gradients (dq, dk, dv) of O = softmax(scale Q K^T) V given dO = dout, in fp64.

    q, dout [B,H,Nq,d]; k, v [B,Hkv,Nk,d] (same dtype code; Hkv divides H and query head h reads
    key/value head h // (H // Hkv); the dk, dv of a key/value head sum over its query heads).
    Causal: key j visible to query i iff j <= i + (Nk - Nq).  P is recomputed from the scores (no stored
    attention matrix), as the backward of the forward definition; see oracle.c for the formulas."""
    qa, code = _as_input(q)
    ka, kcode = _as_input(k)
    va, vcode = _as_input(v)
    da, dcode = _as_input(dout)
    if not (code == kcode == vcode == dcode):
        raise ValueError("q, k, v, dout must share a dtype")
    B, H, Nq, d = qa.shape
    Hkv, Nk = ka.shape[1], ka.shape[2]
    if ka.shape != (B, Hkv, Nk, d) or va.shape != (B, Hkv, Nk, d) or da.shape != (B, H, Nq, d) or H % Hkv:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros((B, H, Nq, d), np.float64)
    dk = np.zeros((B, Hkv, Nk, d), np.float64)
    dv = np.zeros((B, Hkv, Nk, d), np.float64)
    rc = _load().oracle_attn_bwd(_ptr(qa), _ptr(ka), _ptr(va), _ptr(da), code, B, H, Hkv, Nq, Nk, d,
                                 int(bool(causal)), float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _threads(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_bwd failed")
    return dq, dk, dv


def attention_bwd_sampled(q, k, v, dout, q_rows, k_rows, causal=False, scale=None, nthreads=None):
    """The gradients of attention_bwd for ONE head at chosen rows, in fp64, without the [Nq, Nk] matrices:
    q, dout [Nq, d], k, v [Nk, d] (same dtype code); returns dq [len(q_rows), d] and dk, dv [len(k_rows), d]
    at those query / key rows.  Same formulas as attention_bwd; see oracle.c."""
    qa, code = _as_input(q)
    ka, kcode = _as_input(k)
    va, vcode = _as_input(v)
    da, dcode = _as_input(dout)
    if not (code == kcode == vcode == dcode):
        raise ValueError("q, k, v, dout must share a dtype")
    Nq, d = qa.shape
    Nk = ka.shape[0]
    if ka.shape != (Nk, d) or va.shape != (Nk, d) or da.shape != (Nq, d):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    qi = np.ascontiguousarray(np.asarray(q_rows, dtype=np.int64).reshape(-1))
    kj = np.ascontiguousarray(np.asarray(k_rows, dtype=np.int64).reshape(-1))
    dq = np.zeros((qi.size, d), np.float64)
    dk = np.zeros((kj.size, d), np.float64)
    dv = np.zeros((kj.size, d), np.float64)
    rc = _load().oracle_attn_bwd_sampled(_ptr(qa), _ptr(ka), _ptr(va), _ptr(da), code, Nq, Nk, d,
                                         int(bool(causal)), float(scale), _ptr(qi), qi.size, _ptr(kj), kj.size,
                                         _ptr(dq), _ptr(dk), _ptr(dv), _threads(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_bwd_sampled failed")
    return dq, dk, dv


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal=False, scale=None, nthreads=None):
    """Attention over packed sequences, in fp64: q [Tq,H,d], k/v [Tk,Hkv,d] (token-major, same dtype
    code); sequence s is q tokens [cu_q[s], cu_q[s+1]) and k/v tokens [cu_k[s], cu_k[s+1]).  Each
    sequence is the attention() of its own tokens (the per-(b, h) definition above, one batch entry;
    causal: key j visible to query i iff j <= i + (lk - lq) for a sequence of lq queries and lk
    keys, i.e. its queries are its last lq positions).  Only
    slicing and transposes happen here.  Returns (o [Tq,H,d], lse [Tq,H])."""
    qa, _ = _as_input(q)
    ka, _ = _as_input(k)
    va, _ = _as_input(v)
    cq = np.asarray(cu_seqlens_q, dtype=np.int64)
    ck = np.asarray(cu_seqlens_k, dtype=np.int64)
    if cq.shape != ck.shape or cq.ndim != 1 or cq.shape[0] < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must be [num_seqs + 1]")
    Tq, H, d = qa.shape
    o = np.zeros((Tq, H, d), np.float64)
    lse = np.full((Tq, H), -np.inf, np.float64)
    for s in range(cq.shape[0] - 1):
        q0, q1, k0, k1 = int(cq[s]), int(cq[s + 1]), int(ck[s]), int(ck[s + 1])
        if q1 <= q0:
            continue
        qs = np.ascontiguousarray(qa[q0:q1].transpose(1, 0, 2)[None])
        ks = np.ascontiguousarray(ka[k0:k1].transpose(1, 0, 2)[None])
        vs = np.ascontiguousarray(va[k0:k1].transpose(1, 0, 2)[None])
        os_, ls_ = attention(qs, ks, vs, causal=causal, scale=scale, nthreads=nthreads)
        o[q0:q1] = os_[0].transpose(1, 0, 2)
        lse[q0:q1] = ls_[0].T
    return o, lse


def attention_bwd_varlen(q, k, v, dout, cu_seqlens_q, cu_seqlens_k, causal=False, scale=None, nthreads=None):
    """The gradients of attention_varlen, in fp64: q, dout [Tq,H,d], k/v [Tk,Hkv,d] token-major (same dtype
    code).  Each sequence's tokens get the attention_bwd of that sequence alone (a sequence without keys has
    a constant output, so zero gradients; keys no query sees get zero).  Only slicing and transposes happen
    here.  Returns (dq [Tq,H,d], dk [Tk,Hkv,d], dv [Tk,Hkv,d])."""
    qa, _ = _as_input(q)
    ka, _ = _as_input(k)
    va, _ = _as_input(v)
    da, _ = _as_input(dout)
    cq = np.asarray(cu_seqlens_q, dtype=np.int64)
    ck = np.asarray(cu_seqlens_k, dtype=np.int64)
    if cq.shape != ck.shape or cq.ndim != 1 or cq.shape[0] < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must be [num_seqs + 1]")
    dq = np.zeros(qa.shape, np.float64)
    dk = np.zeros(ka.shape, np.float64)
    dv = np.zeros(va.shape, np.float64)
    heads_first = lambda a: np.ascontiguousarray(a.transpose(1, 0, 2)[None])
    for s in range(cq.shape[0] - 1):
        q0, q1, k0, k1 = int(cq[s]), int(cq[s + 1]), int(ck[s]), int(ck[s + 1])
        if q1 <= q0 or k1 <= k0:
            continue
        g = attention_bwd(heads_first(qa[q0:q1]), heads_first(ka[k0:k1]), heads_first(va[k0:k1]),
                          heads_first(da[q0:q1]), causal=causal, scale=scale, nthreads=nthreads)
        dq[q0:q1] = g[0][0].transpose(1, 0, 2)
        dk[k0:k1] = g[1][0].transpose(1, 0, 2)
        dv[k0:k1] = g[2][0].transpose(1, 0, 2)
    return dq, dk, dv


def lse_merge(part_o, part_lse):
    """Merge split partials (normalised o_c [S,R,d], lse_c [S,R]) into (o [R,d], lse [R])."""
    pl = np.ascontiguousarray(np.asarray(part_lse, np.float64))
    S, R = pl.shape
    if part_o is None:
        d = 0
        po = None
    else:
        po = np.ascontiguousarray(np.asarray(part_o, np.float64))
        d = po.shape[2]
        if po.shape[:2] != (S, R):
            raise ValueError("part_o must be [S,R,d]")
    o = np.zeros((R, d), np.float64)
    lse = np.empty(R, np.float64)
    rc = _load().oracle_lse_merge(_ptr(po), _ptr(pl), S, R, d, _ptr(o) if d > 0 else None, _ptr(lse))
    if rc != 0:
        raise RuntimeError("oracle_lse_merge failed")
    return o, lse


def online_stats(x):
    """Single-pass running (m, l) over a 1-D array (the element-by-element scan)."""
    xa = np.ascontiguousarray(np.asarray(x, np.float64).reshape(-1))
    m, l = ctypes.c_double(), ctypes.c_double()
    _load().oracle_online_stats(_ptr(xa), xa.shape[0], ctypes.byref(m), ctypes.byref(l))
    return m.value, l.value


def online_stats_trace(x):
    """(m_k, d_k) after each element of the scan, as two arrays."""
    xa = np.ascontiguousarray(np.asarray(x, np.float64).reshape(-1))
    ms = np.empty_like(xa)
    ls = np.empty_like(xa)
    _load().oracle_online_stats_trace(_ptr(xa), xa.shape[0], _ptr(ms), _ptr(ls))
    return ms, ls


def merge_ml(m1, l1, m2, l2):
    """Merge two (m, l) segment statistics; 0 is the reference when both maxima are -inf."""
    m, l = ctypes.c_double(), ctypes.c_double()
    _load().oracle_merge_ml(float(m1), float(l1), float(m2), float(l2), ctypes.byref(m), ctypes.byref(l))
    return m.value, l.value


def attention_fa1(q, k, v, Br=4, Bc=3, scale=None):
    """FlashAttention V1 block order for one head (non-causal), fp64: q [N,d], k/v [Nk,d]."""
    qa = np.ascontiguousarray(np.asarray(q, np.float64))
    ka = np.ascontiguousarray(np.asarray(k, np.float64))
    va = np.ascontiguousarray(np.asarray(v, np.float64))
    N, d = qa.shape
    Nk = ka.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((N, d), np.float64)
    rc = _load().oracle_attn_fa1(_ptr(qa), _ptr(ka), _ptr(va), N, Nk, d, Br, Bc, float(scale), _ptr(o))
    if rc != 0:
        raise RuntimeError("oracle_attn_fa1 failed")
    return o
