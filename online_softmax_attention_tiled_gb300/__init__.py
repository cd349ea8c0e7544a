"""Python binding of the online-softmax tiled attention library for GB300.

A thin ctypes layer over ``liboa.so`` (the C ABI in ``include/oa.h``): it
allocates output tensors with PyTorch, passes device pointers, sizes and the
current CUDA stream, and turns status codes into exceptions.  Every step of
the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback -- if the library is missing or cannot load, calls raise.

Entry points (same names as the C ABI, without the ``oa_`` prefix):
  softmax_rows, attn_fwd, attn_fwd_f32_tiles, attn_splitkv,
  splitkv_workspace_bytes, attn_splitkv_static, lse_merge, sync_status, set_wait_limit_ns,
  selftest_wait_timeout, selftest_debug_check.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# OA_DEBUG=1 in the environment loads the debug build (bounds and alignment checks in the kernels,
# recorded in the status word that sync_status reads) instead of the release library.
DEBUG = os.environ.get("OA_DEBUG", "") == "1"
LIB_PATH = os.path.join(_PKG, "liboa_debug.so" if DEBUG else "liboa.so")

OA_OK, OA_ERR_INVALID, OA_ERR_UNSUPPORTED, OA_ERR_CUDA, OA_ERR_TIMEOUT = 0, 1, 2, 3, 4
OA_F32, OA_BF16 = 0, 1

EXPORTS = (
    "oa_status_string", "oa_last_error", "oa_version", "oa_softmax_rows", "oa_attn_fwd", "oa_attn_fwd_gqa",
    "oa_attn_fwd_varlen", "oa_attn_fwd_f32_tiles", "oa_splitkv_workspace_bytes", "oa_attn_splitkv",
    "oa_attn_splitkv_gqa", "oa_attn_splitkv_static", "oa_lse_merge", "oa_attn_bwd_workspace_bytes", "oa_attn_bwd",
    "oa_attn_fwd_host_workspace_bytes", "oa_attn_fwd_host", "oa_attn_bwd_gqa", "oa_attn_bwd_varlen",
    "oa_sync_status", "oa_set_wait_limit_ns", "oa_selftest_wait_timeout", "oa_selftest_debug_check",
)


class OAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def _status_name(s):
    return {0: "OA_OK", 1: "OA_ERR_INVALID", 2: "OA_ERR_UNSUPPORTED", 3: "OA_ERR_CUDA",
            4: "OA_ERR_TIMEOUT"}.get(s, f"status {s}")


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load liboa.so (building it with nvcc first if it is absent).  Raises if it cannot."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            if not build_if_missing:
                raise RuntimeError(f"CUDA library not built: {LIB_PATH}")
            from ._build import build

            build(debug=DEBUG)
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, f32, u64, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                      ctypes.c_uint64, ctypes.c_size_t)
        sig = {
            "oa_status_string": ([i32], ctypes.c_char_p),
            "oa_last_error": ([], ctypes.c_char_p),
            "oa_version": ([], i32),
            "oa_softmax_rows": ([vp, i64, i64, i64, vp, i64, vp, vp], i32),
            "oa_attn_fwd": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp, vp], i32),
            "oa_attn_fwd_gqa": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, vp, vp], i32),
            "oa_attn_fwd_varlen": ([vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                    f32, vp], i32),
            "oa_attn_fwd_f32_tiles": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, i32, i32, vp],
                                      i32),
            "oa_splitkv_workspace_bytes": ([i32, i32, i32, i32, i32], sz),
            "oa_attn_splitkv": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, i32, vp, sz, vp], i32),
            "oa_attn_splitkv_gqa": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp, i32, vp, sz, vp],
                                    i32),
            "oa_attn_splitkv_static": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, vp, i32, vp], i32),
            "oa_lse_merge": ([vp, vp, i32, i64, i32, vp, i32, vp, vp], i32),
            "oa_attn_bwd_workspace_bytes": ([i32, i32, i32, i32], sz),
            "oa_attn_fwd_host_workspace_bytes": ([i32, i32, i32, i32, i32, i32, i32], sz),
            "oa_attn_bwd_gqa": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, vp,
                                 sz, vp], i32),
            "oa_attn_bwd_varlen": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                    i32, i32, f32, vp, sz, vp], i32),
            "oa_attn_fwd_host": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp],
                                 i32),
            "oa_attn_bwd": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp],
                            i32),
            "oa_sync_status": ([vp], i32),
            "oa_set_wait_limit_ns": ([u64], None),
            "oa_selftest_wait_timeout": ([u64, vp], i32),
            "oa_selftest_debug_check": ([vp, vp], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(status: int):
    if status != OA_OK:
        msg = load().oa_last_error().decode(errors="replace")
        raise OAError(status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(dt):
    if dt == torch.float32:
        return OA_F32
    if dt == torch.bfloat16:
        return OA_BF16
    raise OAError(OA_ERR_UNSUPPORTED, f"dtype {dt} (need float32 or bfloat16)")


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise OAError(OA_ERR_INVALID, "tensors must live on a CUDA device")


def _same_device(device, *ts):
    for t in ts:
        if t is not None and t.device != device:
            raise OAError(OA_ERR_INVALID, f"every tensor of a call must be on {device} (got one on {t.device})")


def _check_out(t, shape, dtype, device, name):
    """A caller-supplied output must be exactly what the kernel writes: contiguous, of `shape` and
    `dtype`, on `device` (anything else would be written past its end or on another GPU)."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous() or t.device != device:
        raise OAError(OA_ERR_INVALID, f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on "
                      f"{device} (got {t.dtype} {tuple(t.shape)} on {t.device}, "
                      f"{'' if t.is_contiguous() else 'non-'}contiguous)")


def _check_workspace(ws, device):
    if ws is None:
        return
    if ws.device != device or not ws.is_contiguous():
        raise OAError(OA_ERR_INVALID, f"workspace must be a contiguous tensor on {device}")


def version() -> int:
    return load().oa_version()


def softmax_rows(x: torch.Tensor, y: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                 want_y: bool = True, want_lse: bool = True):
    """Row softmax of a 2-D fp32 tensor (unit column stride; any row stride) and per-row LSE.

    Returns (y, lse); either is None when not requested.
    """
    _require_cuda(x, y, lse)
    if x.dim() != 2 or x.dtype != torch.float32 or x.stride(1) != 1:
        raise OAError(OA_ERR_INVALID, "x must be a 2-D float32 tensor with unit column stride")
    rows, cols = x.shape
    if want_y and y is None:
        y = torch.empty((rows, cols), dtype=torch.float32, device=x.device)
    if want_lse and lse is None:
        lse = torch.empty(rows, dtype=torch.float32, device=x.device)
    if y is not None and (y.shape != x.shape or y.stride(1) != 1 or y.dtype != torch.float32 or y.device != x.device
                          or (rows > 1 and y.stride(0) < cols)):
        raise OAError(OA_ERR_INVALID, "y must be a float32 tensor of x's shape on x's device, unit column stride and "
                      "row stride >= cols")
    _check_out(lse, (rows,), torch.float32, x.device, "lse")
    with torch.cuda.device(x.device):
        _check(load().oa_softmax_rows(_ptr(x), rows, cols, x.stride(0), _ptr(y), y.stride(0) if y is not None else 0,
                                      _ptr(lse), _stream(x.device)))
    return y, lse


def _attn_shapes(q, k, v, allow_groups=False):
    """Sizes of q [B, H, Nq, d] and k, v [B, H_kv, Nk, d]; returns (B, H, Nq, Nk, d, H_kv)."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise OAError(OA_ERR_INVALID, "q, k, v must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nk, d) or tuple(v.shape) != (B, Hkv, Nk, d):
        raise OAError(OA_ERR_INVALID, "k and v must be [B, H_kv, Nk, d] matching q")
    if Hkv != H and not (allow_groups and Hkv >= 1 and H % Hkv == 0):
        raise OAError(OA_ERR_INVALID, f"k and v have {Hkv} heads for {H} query heads"
                      + (" (need a divisor of H)" if allow_groups else " (need the same count)"))
    if not (q.dtype == k.dtype == v.dtype):
        raise OAError(OA_ERR_INVALID, "q, k, v must share a dtype")
    _same_device(q.device, k, v)
    for t in (q, k, v):
        if not t.is_contiguous():
            raise OAError(OA_ERR_INVALID, "q, k, v must be contiguous")
    return B, H, Nq, Nk, d, Hkv


def _kv_len_arg(kv_len, B, device):
    if kv_len is None:
        return None
    if kv_len.dtype != torch.int32 or kv_len.shape != (B,) or not kv_len.is_cuda or kv_len.device != device:
        raise OAError(OA_ERR_INVALID, "kv_len must be an int32 CUDA tensor of shape [B] on q's device")
    return kv_len.contiguous()


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, kv_len=None, out=None, lse=None,
             want_lse: bool = True):
    """O = softmax(Q K^T * scale) V with per-row LSE; q [B,H,Nq,d], k/v [B,H_kv,Nk,d] (H_kv divides H;
    query head h reads key/value head h // (H // H_kv)), bf16 or fp32 on CUDA."""
    _require_cuda(q, k, v, out, lse)
    B, H, Nq, Nk, d, Hkv = _attn_shapes(q, k, v, allow_groups=True)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kv = _kv_len_arg(kv_len, B, q.device)
    _check_out(out, (B, H, Nq, d), q.dtype, q.device, "out")
    _check_out(lse, (B, H, Nq), torch.float32, q.device, "lse")
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=q.dtype, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        _check(load().oa_attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _dtype_code(q.dtype), B, H,
                                      Hkv, Nq, Nk, d, int(bool(causal)), float(scale), _ptr(kv), _stream(q.device)))
    return out, lse


def _cu_seqlens_arg(cu, device, name):
    if cu.dtype != torch.int32 or cu.dim() != 1 or cu.numel() < 2 or not cu.is_cuda or cu.device != device:
        raise OAError(OA_ERR_INVALID, f"{name} must be an int32 CUDA tensor of num_seqs + 1 offsets on q's device")
    return cu.contiguous()


def attn_fwd_host_workspace_bytes(dtype, B: int, H: int, H_kv: int, Nq: int, Nk: int, d: int) -> int:
    return int(load().oa_attn_fwd_host_workspace_bytes(_dtype_code(dtype), B, H, H_kv, Nq, Nk, d))


def attn_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, want_lse: bool = True,
                  chunks: int = 0, workspace=None, device=None):
    """attn_fwd on host (CPU) tensors, pinned for the copies to overlap: the library copies q, k, v to the
    device in pieces, runs the forward and copies o and lse back while the next pieces move.  Outputs are
    CPU tensors (pinned when allocated here), complete once the current stream of `device` is synchronised.
    workspace: optional uint8 CUDA tensor of attn_fwd_host_workspace_bytes."""
    for t in (q, k, v, out, lse):
        if t is not None and t.is_cuda:
            raise OAError(OA_ERR_INVALID, "attn_fwd_host takes host tensors")
    B, H, Nq, Nk, d, Hkv = _attn_shapes(q, k, v, allow_groups=True)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=q.dtype).pin_memory()
    if want_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
    if tuple(out.shape) != (B, H, Nq, d) or out.dtype != q.dtype or not out.is_contiguous():
        raise OAError(OA_ERR_INVALID, "out must be a contiguous [B, H, Nq, d] host tensor of q's dtype")
    if lse is not None and (tuple(lse.shape) != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise OAError(OA_ERR_INVALID, "lse must be a contiguous float32 [B, H, Nq] host tensor")
    need = attn_fwd_host_workspace_bytes(q.dtype, B, H, Hkv, Nq, Nk, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _require_cuda(workspace)
    with torch.cuda.device(dev):
        _check(load().oa_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _dtype_code(q.dtype), B, H,
                                       Hkv, Nq, Nk, d, int(bool(causal)), float(scale), int(chunks), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(dev)))
    return out, lse


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                    causal: bool = False, scale: float | None = None, out=None, lse=None, want_lse: bool = True):
    """Attention over packed sequences: q [Tq, H, d], k/v [Tk, H_kv, d] bf16 (token-major); sequence s is
    tokens [cu_seqlens_q[s], cu_seqlens_q[s+1]) of q and [cu_seqlens_k[s], cu_seqlens_k[s+1]) of k/v.
    Returns (o [Tq, H, d], lse [Tq, H])."""
    _require_cuda(q, k, v, out, lse)
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise OAError(OA_ERR_INVALID, "q must be [Tq, H, d] and k, v [Tk, H_kv, d]")
    Tq, H, d = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    if tuple(k.shape) != (Tk, Hkv, d) or tuple(v.shape) != (Tk, Hkv, d):
        raise OAError(OA_ERR_INVALID, "k and v must be [Tk, H_kv, d] matching q")
    if not (q.dtype == k.dtype == v.dtype):
        raise OAError(OA_ERR_INVALID, "q, k, v must share a dtype")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise OAError(OA_ERR_INVALID, "q, k, v must be contiguous")
    cq = _cu_seqlens_arg(cu_seqlens_q, q.device, "cu_seqlens_q")
    ck = _cu_seqlens_arg(cu_seqlens_k, q.device, "cu_seqlens_k")
    if cq.numel() != ck.numel():
        raise OAError(OA_ERR_INVALID, "cu_seqlens_q and cu_seqlens_k must have the same length")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _same_device(q.device, k, v)
    _check_out(out, (Tq, H, d), q.dtype, q.device, "out")
    _check_out(lse, (Tq, H), torch.float32, q.device, "lse")
    if out is None:
        out = torch.empty((Tq, H, d), dtype=q.dtype, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((Tq, H), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        _check(load().oa_attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _dtype_code(q.dtype),
                                         _ptr(cq), _ptr(ck), cq.numel() - 1, H, Hkv, Tq, Tk, int(max_seqlen_q),
                                         int(max_seqlen_k), d, int(bool(causal)), float(scale), _stream(q.device)))
    return out, lse


def attn_fwd_f32_tiles(q, k, v, Br: int, Bc: int, causal: bool = False, scale: float | None = None, kv_len=None,
                       out=None, lse=None):
    """fp32 attention forward with explicit tile sizes (Br query rows, Bc keys per step)."""
    _require_cuda(q, k, v, out, lse)
    B, H, Nq, Nk, d, Hkv = _attn_shapes(q, k, v)
    if q.dtype != torch.float32:
        raise OAError(OA_ERR_INVALID, "attn_fwd_f32_tiles needs float32 inputs")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kv = _kv_len_arg(kv_len, B, q.device)
    _check_out(out, (B, H, Nq, d), q.dtype, q.device, "out")
    _check_out(lse, (B, H, Nq), torch.float32, q.device, "lse")
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        _check(load().oa_attn_fwd_f32_tiles(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, d,
                                            int(bool(causal)), float(scale), _ptr(kv), int(Br), int(Bc),
                                            _stream(q.device)))
    return out, lse


def attn_bwd_workspace_bytes(B: int, H: int, Nq: int, d: int) -> int:
    return int(load().oa_attn_bwd_workspace_bytes(B, H, Nq, d))


def attn_bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
             workspace=None):
    """Gradients (dq, dk, dv) of O = softmax(Q K^T * scale) V for the upstream gradient dout, with P recomputed
    from the forward's LSE.  q, o, dout [B,H,Nq,d] and k, v [B,H_kv,Nk,d] (H_kv divides H: grouped key/value
    heads, whose dk, dv sum over their query heads), bf16 on CUDA; lse fp32 [B,H,Nq] (o and lse from attn_fwd
    on the same inputs).  workspace: optional uint8 CUDA tensor of attn_bwd_workspace_bytes."""
    _require_cuda(q, k, v, o, lse, dout, dq, dk, dv, workspace)
    B, H, Nq, Nk, d, Hkv = _attn_shapes(q, k, v, allow_groups=True)
    if tuple(o.shape) != (B, H, Nq, d) or tuple(dout.shape) != (B, H, Nq, d):
        raise OAError(OA_ERR_INVALID, "o and dout must be [B, H, Nq, d] like q")
    if o.dtype != q.dtype or dout.dtype != q.dtype or not o.is_contiguous() or not dout.is_contiguous():
        raise OAError(OA_ERR_INVALID, "o and dout must be contiguous with q's dtype")
    if lse is None or tuple(lse.shape) != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise OAError(OA_ERR_INVALID, "lse must be a contiguous float32 [B, H, Nq] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _same_device(q.device, o, lse, dout)
    _check_out(dq, (B, H, Nq, d), q.dtype, q.device, "dq")
    _check_out(dk, (B, Hkv, Nk, d), q.dtype, q.device, "dk")
    _check_out(dv, (B, Hkv, Nk, d), q.dtype, q.device, "dv")
    _check_workspace(workspace, q.device)
    need = attn_bwd_workspace_bytes(B, H, Nq, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    with torch.cuda.device(q.device):
        _check(load().oa_attn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                                      _ptr(dk), _ptr(dv), _dtype_code(q.dtype), B, H, Hkv, Nq, Nk, d,
                                      int(bool(causal)), float(scale), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(q.device)))
    return dq, dk, dv


def attn_bwd_varlen(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                    causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None, workspace=None):
    """Gradients of attn_fwd_varlen: q, o, dout [Tq, H, d] and k, v [Tk, H_kv, d] bf16 (token-major), lse fp32
    [Tq, H] from attn_fwd_varlen on the same inputs.  Returns (dq, dk, dv) in the layouts of q, k, v."""
    _require_cuda(q, k, v, o, lse, dout, dq, dk, dv, workspace)
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise OAError(OA_ERR_INVALID, "q must be [Tq, H, d] and k, v [Tk, H_kv, d]")
    Tq, H, d = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    if tuple(k.shape) != (Tk, Hkv, d) or tuple(v.shape) != (Tk, Hkv, d):
        raise OAError(OA_ERR_INVALID, "k and v must be [Tk, H_kv, d] matching q")
    for t in (q, k, v, o, dout):
        if t.dtype != q.dtype or not t.is_contiguous():
            raise OAError(OA_ERR_INVALID, "q, k, v, o, dout must be contiguous with one dtype")
    if tuple(o.shape) != (Tq, H, d) or tuple(dout.shape) != (Tq, H, d):
        raise OAError(OA_ERR_INVALID, "o and dout must be [Tq, H, d] like q")
    if lse is None or tuple(lse.shape) != (Tq, H) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise OAError(OA_ERR_INVALID, "lse must be a contiguous float32 [Tq, H] tensor")
    cq = _cu_seqlens_arg(cu_seqlens_q, q.device, "cu_seqlens_q")
    ck = _cu_seqlens_arg(cu_seqlens_k, q.device, "cu_seqlens_k")
    if cq.numel() != ck.numel():
        raise OAError(OA_ERR_INVALID, "cu_seqlens_q and cu_seqlens_k must have the same length")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _same_device(q.device, k, v, o, lse, dout)
    _check_out(dq, (Tq, H, d), q.dtype, q.device, "dq")
    _check_out(dk, (Tk, Hkv, d), q.dtype, q.device, "dk")
    _check_out(dv, (Tk, Hkv, d), q.dtype, q.device, "dv")
    _check_workspace(workspace, q.device)
    need = attn_bwd_workspace_bytes(1, H, Tq, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    with torch.cuda.device(q.device):
        _check(load().oa_attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                                         _ptr(dk), _ptr(dv), _dtype_code(q.dtype), _ptr(cq), _ptr(ck), cq.numel() - 1,
                                         H, Hkv, Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), d, int(bool(causal)),
                                         float(scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(q.device)))
    return dq, dk, dv


def splitkv_workspace_bytes(B: int, H: int, Nq: int, d: int, num_splits: int) -> int:
    return int(load().oa_splitkv_workspace_bytes(B, H, Nq, d, num_splits))


def attn_splitkv(q, k, v, num_splits: int, scale: float | None = None, kv_len=None, out=None, lse=None,
                 workspace=None):
    """Split-KV attention: per-chunk partials, then the LSE merge.  q [B,H,Nq,d], k/v [B,H_kv,Nk,d] (H_kv
    divides H: grouped key/value heads, e.g. a KV cache with fewer heads).  workspace: optional uint8 CUDA
    tensor."""
    _require_cuda(q, k, v, out, lse, workspace)
    B, H, Nq, Nk, d, Hkv = _attn_shapes(q, k, v, allow_groups=True)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kv = _kv_len_arg(kv_len, B, q.device)
    _check_out(out, (B, H, Nq, d), q.dtype, q.device, "out")
    _check_out(lse, (B, H, Nq), torch.float32, q.device, "lse")
    _check_workspace(workspace, q.device)
    need = splitkv_workspace_bytes(B, H, Nq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        _check(load().oa_attn_splitkv_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _dtype_code(q.dtype),
                                          B, H, Hkv, Nq, Nk, d, float(scale), _ptr(kv), int(num_splits),
                                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(q.device)))
    return out, lse


def attn_splitkv_static(q, k, v, num_splits: int, scale: float | None = None, kv_len=None, out=None, lse=None):
    """Split-KV attention whose partials live in the library's fixed 16 MiB device scratch (no
    workspace).  For callers that cannot allocate device memory at call time: pass `out` and `lse`
    to allocate nothing here either.  Calls that overlap on the GPU share the scratch and race."""
    _require_cuda(q, k, v, out, lse)
    B, H, Nq, Nk, d, Hkv = _attn_shapes(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kv = _kv_len_arg(kv_len, B, q.device)
    _check_out(out, (B, H, Nq, d), q.dtype, q.device, "out")
    _check_out(lse, (B, H, Nq), torch.float32, q.device, "lse")
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        _check(load().oa_attn_splitkv_static(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _dtype_code(q.dtype),
                                             B, H, Nq, Nk, d, float(scale), _ptr(kv), int(num_splits),
                                             _stream(q.device)))
    return out, lse


def lse_merge(part_o, part_lse, out_dtype=torch.float32, out=None, lse=None):
    """Merge S partials: part_o fp32 [S, R, d] (or None for d = 0), part_lse fp32 [S, R]."""
    _require_cuda(part_o, part_lse, out, lse)
    if part_lse.dim() != 2 or part_lse.dtype != torch.float32 or not part_lse.is_contiguous():
        raise OAError(OA_ERR_INVALID, "part_lse must be a contiguous float32 [S, R] tensor")
    S, R = part_lse.shape
    d = 0
    if part_o is not None:
        if part_o.dim() != 3 or tuple(part_o.shape[:2]) != (S, R) or part_o.dtype != torch.float32 or \
                not part_o.is_contiguous():
            raise OAError(OA_ERR_INVALID, "part_o must be a contiguous float32 [S, R, d] tensor")
        d = part_o.shape[2]
        _same_device(part_lse.device, part_o)
    if out is not None:
        if d == 0:
            raise OAError(OA_ERR_INVALID, "out is only written when part_o is given")
        _check_out(out, (R, d), out.dtype, part_lse.device, "out")
        _dtype_code(out.dtype)
    _check_out(lse, (R,), torch.float32, part_lse.device, "lse")
    if d > 0 and out is None:
        out = torch.empty((R, d), dtype=out_dtype, device=part_lse.device)
    if lse is None:
        lse = torch.empty(R, dtype=torch.float32, device=part_lse.device)
    code = _dtype_code(out.dtype if out is not None else out_dtype)
    with torch.cuda.device(part_lse.device):
        _check(load().oa_lse_merge(_ptr(part_o), _ptr(part_lse), S, R, d, _ptr(out), code, _ptr(lse),
                                   _stream(part_lse.device)))
    return out, lse


def sync_status(device=None):
    """Synchronise the current stream and raise OAError if a device wait expired."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(load().oa_sync_status(_stream(dev)))


def set_wait_limit_ns(ns: int):
    load().oa_set_wait_limit_ns(int(ns))


def selftest_wait_timeout(limit_ns: int = 1_000_000, device=None):
    """Launch a wait that nothing satisfies; it must give up after limit_ns (see oa.h)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(load().oa_selftest_wait_timeout(int(limit_ns), _stream(dev)))


def selftest_debug_check(device=None) -> int:
    """Launch one store guarded by a failing debug check (see oa.h); returns the flag it guards (0 when
    the debug build skipped the store, 1 in the release build).  The caller reads the check's report
    with sync_status()."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(load().oa_selftest_debug_check(flag.data_ptr(), _stream(dev)))
        torch.cuda.current_stream(dev).synchronize()
    return int(flag.item())
