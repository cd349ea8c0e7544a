"""The allocation-free split-KV entry point, oa_attn_splitkv_static, through the C ABI.

Some callers cannot allocate device memory when they call: an application that owns
all device memory through its own allocator and hands the library only its inputs and
outputs, or a latency-critical decode loop where a cudaMalloc could block or fail.
oa_attn_splitkv_static keeps its per-chunk partials in a 16 MiB array inside the
library instead of a caller workspace.  These tests check, on two calls in a row with
different inputs and cache lengths, that its output matches the workspace entry point
(oa_attn_splitkv) and the fp64 CPU oracle within the tolerances of the other tests, and
that the second call leaves the device's free memory unchanged.  Each test builds its
own inputs, so it passes alone in a fresh process or after the rest of the suite; the
file name only makes it run last.
"""
import pytest
import torch

import oracle
import synth_inputs as si
from parity import BF16_O_ATOL, LSE_ATOL, assert_lse_close, assert_out_close, bf16_bits, to_np

pytestmark = pytest.mark.gpu

SHAPE = dict(B=4, H=8, Nq=2, Nk=3000, d=128)


def _inputs(seed):
    s = SHAPE
    return si.attn_inputs(s["B"], s["H"], s["Nq"], s["Nk"], s["d"], torch.bfloat16, seed=seed)


def test_static_scratch_matches_workspace_entry_point_and_oracle(cuda_lib):
    oa = cuda_lib
    splits = 24  # needs 24 * 64 rows * 129 * 4 B = 792 KB of the 16 MiB scratch
    out = torch.empty((4, 8, 2, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((4, 8, 2), dtype=torch.float32, device="cuda")
    for call, (seed, kv) in enumerate([(10, [3000, 1, 0, 1777]), (11, [0, 2999, 3000, 512])]):
        q, k, v = _inputs(seed)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        kv_len = torch.tensor(kv, dtype=torch.int32, device="cuda")
        ref_o, ref_lse = oa.attn_splitkv(qd, kd, vd, splits, kv_len=kv_len)
        out.fill_(7.0)  # stale values must be overwritten
        lse.fill_(7.0)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        oa.attn_splitkv_static(qd, kd, vd, splits, kv_len=kv_len, out=out, lse=lse)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        oa.sync_status()
        if call == 1:  # the first call on a device loads the scratch; later calls allocate nothing
            assert free_after == free_before, f"device free memory changed by {free_before - free_after} bytes"
        # against the workspace entry point
        assert_lse_close(lse, to_np(ref_lse), LSE_ATOL, what=f"lse vs workspace path (call {call})")
        assert_out_close(out, to_np(ref_o), BF16_O_ATOL, lse_ref=to_np(ref_lse), what=f"O vs workspace (call {call})")
        # against the fp64 oracle
        oo, ol = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), kv_len=kv)
        assert_lse_close(lse, ol, LSE_ATOL, what=f"lse vs oracle (call {call})")
        assert_out_close(out, oo, BF16_O_ATOL, lse_ref=ol, what=f"O vs oracle (call {call})")


def test_static_scratch_rejects_oversized_requests(cuda_lib):
    oa = cuda_lib
    q, k, v = si.attn_inputs(32, 32, 1, 1024, 128, torch.bfloat16, seed=1, device="cuda")
    # 64 * 1024 rows * 129 * 4 B = 33.8 MB > 16 MiB
    with pytest.raises(oa.OAError) as ei:
        oa.attn_splitkv_static(q, k, v, 64)
    assert ei.value.status == oa.OA_ERR_INVALID
    assert "16 MiB" in str(ei.value)
