"""Host-side checks of the C ABI: no GPU needed, no kernel is launched.

The library must load, export every function include/oa.h declares, and
reject invalid arguments on the host (these calls return before any CUDA
call).  Valid compute calls are left to the gpu-marked tests.
"""
import ctypes
import os
import re

import pytest

import online_softmax_attention_tiled_gb300 as oa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "oa.h")
FAKE = ctypes.c_void_p(0x10000)  # 64 KiB-aligned, never dereferenced on the host
FAKE_ODD = ctypes.c_void_p(0x10002)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return oa.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in oa.h but not exported"
    assert set(names) == set(oa.EXPORTS)


def test_status_strings_and_version(lib):
    for s in range(5):
        assert lib.oa_status_string(s).startswith(b"OA_")
    assert lib.oa_status_string(99) == b"unknown oa_status"
    assert lib.oa_version() >= 100


def test_workspace_size_formula(lib):
    # num_splits * rows * (d + 1) fp32 values, rounded up to 256 bytes
    b = lib.oa_splitkv_workspace_bytes(32, 32, 1, 128, 64)
    assert b == ((64 * 32 * 32 * 129 * 4 + 255) // 256) * 256
    assert lib.oa_splitkv_workspace_bytes(0, 1, 1, 1, 1) == 0
    assert lib.oa_splitkv_workspace_bytes(1, 1, 1, 1, 0) == 0


def _err(lib):
    return lib.oa_last_error().decode()


def test_softmax_rows_validation(lib):
    NULL = None
    assert lib.oa_softmax_rows(NULL, 4, 4, 4, FAKE, 4, FAKE, NULL) == oa.OA_ERR_INVALID
    assert "x is NULL" in _err(lib)
    assert lib.oa_softmax_rows(FAKE, 0, 4, 4, FAKE, 4, FAKE, NULL) == oa.OA_ERR_INVALID
    assert lib.oa_softmax_rows(FAKE, 4, 0, 4, FAKE, 4, FAKE, NULL) == oa.OA_ERR_INVALID
    assert lib.oa_softmax_rows(FAKE, 4, 8, 4, FAKE, 8, FAKE, NULL) == oa.OA_ERR_INVALID  # ld_x < cols
    assert lib.oa_softmax_rows(FAKE, 4, 8, 8, FAKE, 4, FAKE, NULL) == oa.OA_ERR_INVALID  # ld_y < cols
    assert lib.oa_softmax_rows(FAKE, 4, 8, 8, NULL, 8, NULL, NULL) == oa.OA_ERR_INVALID  # no output
    assert lib.oa_softmax_rows(FAKE_ODD, 4, 8, 8, FAKE, 8, FAKE, NULL) == oa.OA_ERR_INVALID  # misaligned
    assert lib.oa_softmax_rows(FAKE, 4, 8, 8, FAKE, 16, NULL, NULL) == oa.OA_ERR_INVALID  # in place, ld differs


def test_attn_fwd_validation(lib):
    NULL = None
    args = dict(B=1, H=1, Nq=8, Nk=8, d=64, causal=0, scale=0.125)

    def call(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dt=oa.OA_BF16, **kw):
        a = dict(args, **kw)
        return lib.oa_attn_fwd(q, k, v, o, lse, dt, a["B"], a["H"], a["Nq"], a["Nk"], a["d"], a["causal"],
                               a["scale"], NULL, NULL)

    assert call(q=NULL) == oa.OA_ERR_INVALID
    assert call(o=NULL) == oa.OA_ERR_INVALID
    assert call(B=0) == oa.OA_ERR_INVALID
    assert call(Nk=0) == oa.OA_ERR_INVALID
    assert call(scale=0.0) == oa.OA_ERR_INVALID
    assert call(scale=float("nan")) == oa.OA_ERR_INVALID
    assert call(scale=float("inf")) == oa.OA_ERR_INVALID
    assert call(causal=2) == oa.OA_ERR_INVALID
    assert call(q=FAKE_ODD) == oa.OA_ERR_INVALID
    assert call(dt=7) == oa.OA_ERR_INVALID
    assert call(d=96) == oa.OA_ERR_UNSUPPORTED  # bf16 tensor-core path: d in {64, 128}
    assert "d = 64 or 128" in _err(lib)
    assert call(dt=oa.OA_F32, d=300) == oa.OA_ERR_UNSUPPORTED


def test_attn_fwd_f32_tiles_validation(lib):
    NULL = None
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 6, 6, 4, 0, 0.5, NULL]
    assert lib.oa_attn_fwd_f32_tiles(*base, 0, 3, NULL) == oa.OA_ERR_INVALID
    assert lib.oa_attn_fwd_f32_tiles(*base, 4, 65, NULL) == oa.OA_ERR_INVALID
    big = [FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 6, 6, 256, 0, 0.5, NULL]
    assert lib.oa_attn_fwd_f32_tiles(*big, 64, 64, NULL) == oa.OA_ERR_UNSUPPORTED  # > 227 KB of smem


def test_attn_splitkv_validation(lib):
    NULL = None
    need = lib.oa_splitkv_workspace_bytes(2, 2, 1, 128, 4)

    def call(dt=oa.OA_BF16, d=128, splits=4, ws=FAKE, ws_bytes=need):
        return lib.oa_attn_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, dt, 2, 2, 1, 64, d, 0.1, NULL, splits, ws, ws_bytes,
                                   NULL)

    assert call(ws=NULL) == oa.OA_ERR_INVALID
    assert call(ws_bytes=need - 1) == oa.OA_ERR_INVALID
    assert call(ws=FAKE_ODD) == oa.OA_ERR_INVALID
    assert call(splits=0) == oa.OA_ERR_INVALID
    assert call(splits=1025) == oa.OA_ERR_INVALID
    assert call(d=96) == oa.OA_ERR_UNSUPPORTED
    assert call(dt=oa.OA_F32, d=256) == oa.OA_ERR_UNSUPPORTED


def test_attn_bwd_validation(lib):
    NULL = None
    need = lib.oa_attn_bwd_workspace_bytes(2, 2, 100, 64)
    assert need == ((2 * 2 * 100 * 65 * 4 + 255) // 256) * 256
    assert lib.oa_attn_bwd_workspace_bytes(0, 2, 100, 64) == 0

    def call(q=FAKE, o=FAKE, dout=FAKE, lse=FAKE, dk=FAKE, dt=oa.OA_BF16, Nq=100, Nk=100, d=64, causal=1,
             scale=0.125, ws=FAKE, ws_bytes=need):
        return lib.oa_attn_bwd(q, FAKE, FAKE, o, dout, lse, FAKE, dk, FAKE, dt, 2, 2, Nq, Nk, d, causal, scale, ws,
                               ws_bytes, NULL)

    for bad in (dict(q=NULL), dict(o=NULL), dict(dout=NULL), dict(lse=NULL), dict(dk=NULL), dict(Nq=0),
                dict(scale=-1.0), dict(causal=3), dict(dout=FAKE_ODD), dict(ws=NULL), dict(ws=FAKE_ODD),
                dict(ws_bytes=need - 1)):
        assert call(**bad) == oa.OA_ERR_INVALID, bad
    assert call(dt=oa.OA_F32) == oa.OA_ERR_UNSUPPORTED
    assert call(d=96) == oa.OA_ERR_UNSUPPORTED
    assert "d = 64 or 128" in _err(lib)
    # packed sequences: the offsets are required, and max_seqlen_k must lie in [1, total_k]
    assert lib.oa_attn_bwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, oa.OA_BF16, NULL, FAKE, 2, 2, 2,
                                  100, 100, 50, 50, 64, 1, 0.125, FAKE, need, NULL) == oa.OA_ERR_INVALID
    assert lib.oa_attn_bwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, oa.OA_BF16, FAKE, FAKE, 2, 2, 2,
                                  100, 100, 50, 101, 64, 1, 0.125, FAKE, need, NULL) == oa.OA_ERR_INVALID
    # grouped heads: H_kv must divide H
    assert lib.oa_attn_bwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, oa.OA_BF16, 2, 2, 3, 100, 100, 64,
                               1, 0.125, FAKE, need, NULL) == oa.OA_ERR_INVALID


def test_attn_fwd_host_validation(lib):
    NULL = None
    need = lib.oa_attn_fwd_host_workspace_bytes(oa.OA_BF16, 2, 8, 2, 100, 100, 64)
    r = lambda n: (n + 255) // 256 * 256
    assert need == 2 * r(2 * 8 * 100 * 64 * 2) + 2 * r(2 * 2 * 100 * 64 * 2) + r(2 * 8 * 100 * 4)
    assert lib.oa_attn_fwd_host_workspace_bytes(7, 2, 8, 2, 100, 100, 64) == 0
    WS = ctypes.c_void_p(0x100000)

    def call(q=FAKE, o=FAKE, dt=oa.OA_BF16, H=8, Hkv=2, d=64, causal=1, Nk=100, chunks=0, ws=WS, ws_bytes=need):
        return lib.oa_attn_fwd_host(q, FAKE, FAKE, o, FAKE, dt, 2, H, Hkv, 100, Nk, d, causal, 0.125, chunks, ws,
                                    ws_bytes, NULL)

    for bad in (dict(q=NULL), dict(o=NULL), dict(q=FAKE_ODD), dict(Hkv=3), dict(causal=2), dict(chunks=-1),
                dict(chunks=65), dict(ws=NULL), dict(ws=ctypes.c_void_p(0x100010)), dict(ws_bytes=need - 1)):
        assert call(**bad) == oa.OA_ERR_INVALID, bad
    assert call(d=96) == oa.OA_ERR_UNSUPPORTED


def test_lse_merge_validation(lib):
    NULL = None
    assert lib.oa_lse_merge(FAKE, NULL, 2, 4, 8, FAKE, oa.OA_F32, FAKE, NULL) == oa.OA_ERR_INVALID
    assert lib.oa_lse_merge(FAKE, FAKE, 0, 4, 8, FAKE, oa.OA_F32, FAKE, NULL) == oa.OA_ERR_INVALID
    assert lib.oa_lse_merge(FAKE, FAKE, 2, 0, 8, FAKE, oa.OA_F32, FAKE, NULL) == oa.OA_ERR_INVALID
    assert lib.oa_lse_merge(NULL, FAKE, 2, 4, 8, FAKE, oa.OA_F32, FAKE, NULL) == oa.OA_ERR_INVALID
    assert lib.oa_lse_merge(NULL, FAKE, 2, 4, 0, NULL, oa.OA_F32, NULL, NULL) == oa.OA_ERR_INVALID
    assert lib.oa_lse_merge(FAKE, FAKE, 2, 4, 8, FAKE, 5, FAKE, NULL) == oa.OA_ERR_INVALID


def test_selftest_limit_validation(lib):
    assert lib.oa_selftest_wait_timeout(10, None) == oa.OA_ERR_INVALID
    assert lib.oa_selftest_wait_timeout(10 ** 11, None) == oa.OA_ERR_INVALID


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """The product path has no fallback: a missing library is an error."""
    monkeypatch.setattr(oa, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(oa, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        oa.load(build_if_missing=False)


def test_product_package_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "online_softmax_attention_tiled_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle.c" not in text and "liboa_oracle" not in text, f


def test_binding_rejects_mismatched_outputs_before_any_launch():
    """The wrappers check caller-supplied outputs (shape, dtype, contiguity, device) before calling
    the library: a wrong `out` would otherwise be written past its end or on another GPU."""
    import torch

    cpu = torch.device("cpu")
    good = torch.empty((2, 3, 5, 8), dtype=torch.bfloat16)
    oa._check_out(None, (2, 3, 5, 8), torch.bfloat16, cpu, "out")
    oa._check_out(good, (2, 3, 5, 8), torch.bfloat16, cpu, "out")
    bad = [
        torch.empty((2, 3, 4, 8), dtype=torch.bfloat16),            # too small
        torch.empty((2, 3, 5, 8), dtype=torch.float32),             # wrong dtype
        torch.empty((2, 3, 8, 5), dtype=torch.bfloat16).transpose(2, 3),  # right shape, not contiguous
    ]
    for t in bad:
        with pytest.raises(oa.OAError) as ei:
            oa._check_out(t, (2, 3, 5, 8), torch.bfloat16, cpu, "out")
        assert ei.value.status == oa.OA_ERR_INVALID
    with pytest.raises(oa.OAError):
        oa._check_out(good, (2, 3, 5, 8), torch.bfloat16, torch.device("cuda", 0), "out")
    with pytest.raises(oa.OAError):
        oa._same_device(torch.device("cuda", 0), good)
    # every device wrapper that takes outputs checks them
    import inspect

    for name in ("attn_fwd", "attn_fwd_varlen", "attn_fwd_f32_tiles", "attn_splitkv", "attn_splitkv_static",
                 "attn_bwd", "attn_bwd_varlen", "lse_merge", "softmax_rows"):
        src = inspect.getsource(getattr(oa, name))
        assert "_check_out(" in src, name
