"""The allocation-free split-KV entry point (oa_attn_splitkv_static) against the
workspace entry point (oa_attn_splitkv), through the C ABI, on two calls in a row.

The allocation-free variant exists for callers that cannot allocate device memory
when they call (an embedding application that owns all device memory, a path where
an allocation could block or fail); its partials live in a 16 MiB array inside the
library.  Outputs are preallocated here so the call itself allocates nothing.
This file is collected last on purpose.
"""
import pytest
import torch

import synth_inputs as si
from parity import BF16_O_ATOL, LSE_ATOL, assert_lse_close, assert_out_close, to_np

pytestmark = pytest.mark.gpu


def _inputs(seed, kv):
    B, H, Nq, Nk, d = 4, 8, 2, 3000, 128
    q, k, v = si.attn_inputs(B, H, Nq, Nk, d, torch.bfloat16, seed=seed, device="cuda")
    kv_len = torch.tensor(kv, dtype=torch.int32, device="cuda")
    return q, k, v, kv_len


def test_static_scratch_matches_workspace_entry_point(cuda_lib):
    oa = cuda_lib
    splits = 24  # needs 24 * 64 rows * 129 * 4 B = 792 KB of the 16 MiB scratch
    out = None
    for call, (seed, kv) in enumerate([(10, [3000, 1, 0, 1777]), (11, [0, 2999, 3000, 512])]):
        q, k, v, kv_len = _inputs(seed, kv)
        ref_o, ref_lse = oa.attn_splitkv(q, k, v, splits, kv_len=kv_len)
        if out is None:
            out = torch.empty_like(q)
            lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
        out.fill_(7.0)  # stale values must be overwritten
        lse.fill_(7.0)
        oa.attn_splitkv_static(q, k, v, splits, kv_len=kv_len, out=out, lse=lse)
        torch.cuda.synchronize()
        oa.sync_status()
        ref_lse_np = to_np(ref_lse)
        assert_lse_close(lse, ref_lse_np, LSE_ATOL, what=f"lse (call {call})")
        assert_out_close(out, to_np(ref_o), BF16_O_ATOL, lse_ref=ref_lse_np, what=f"O (call {call})")


def test_static_scratch_rejects_oversized_requests(cuda_lib):
    oa = cuda_lib
    q, k, v = si.attn_inputs(32, 32, 1, 1024, 128, torch.bfloat16, seed=1, device="cuda")
    # 64 * 1024 rows * 129 * 4 B = 33.8 MB > 16 MiB
    with pytest.raises(oa.OAError) as ei:
        oa.attn_splitkv_static(q, k, v, 64)
    assert ei.value.status == oa.OA_ERR_INVALID
    assert "16 MiB" in str(ei.value)
