"""Split-KV decode attention (partials + LSE merge) vs the fp64 oracle (gpu)."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import BF16_O_ATOL, assert_lse_close, assert_out_close, bf16_bits, to_np

pytestmark = pytest.mark.gpu


def _run(oa, q, k, v, splits, kv_len=None):
    kvd = None if kv_len is None else torch.as_tensor(kv_len, dtype=torch.int32).cuda()
    o, lse = oa.attn_splitkv(q.cuda(), k.cuda(), v.cuda(), splits, kv_len=kvd)
    torch.cuda.synchronize()
    oa.sync_status()
    return o, lse


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [8, 64, 128])
@pytest.mark.parametrize("splits", [1, 3, 64])
def test_small_vs_oracle(cuda_lib, dtype, d, splits):
    B, H, Nq, Nk = 3, 2, 2, 1000
    q, k, v = si.attn_inputs(B, H, Nq, Nk, d, dtype, seed=d + splits)
    kv_len = [1000, 17, 0]
    o, lse = _run(cuda_lib, q, k, v, splits, kv_len)
    if dtype == torch.bfloat16:
        ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), kv_len=kv_len)
        atol = BF16_O_ATOL
    else:
        ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy(), kv_len=kv_len)
        atol = 2e-5
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, atol, lse_ref=rl)


def test_bf16_d256_and_fp32_d4(cuda_lib):
    q, k, v = si.attn_inputs(2, 2, 1, 300, 256, torch.bfloat16, seed=1)
    o, lse = _run(cuda_lib, q, k, v, 5)
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL)
    q, k, v = si.attn_inputs(2, 2, 1, 300, 4, torch.float32, seed=2)
    o, lse = _run(cuda_lib, q, k, v, 7)
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy())
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, 2e-5)


def test_splits_do_not_change_the_result(cuda_lib):
    q, k, v = si.attn_inputs(2, 4, 1, 4096, 128, torch.bfloat16, seed=3)
    o1, l1 = _run(cuda_lib, q, k, v, 1)
    o2, l2 = _run(cuda_lib, q, k, v, 64)
    np.testing.assert_allclose(to_np(o1), to_np(o2), atol=1e-2)
    np.testing.assert_allclose(to_np(l1), to_np(l2), atol=1e-5)


def test_matches_fused_attention(cuda_lib):
    """Split-KV decode and the fused tensor-core kernel agree on the same rows."""
    q, k, v = si.attn_inputs(2, 2, 1, 777, 128, torch.bfloat16, seed=4)
    o1, l1 = _run(cuda_lib, q, k, v, 8)
    o2, l2 = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_np(o1), to_np(o2), atol=2e-2)
    np.testing.assert_allclose(to_np(l1), to_np(l2), atol=1e-4)


@pytest.mark.slow
def test_full_size_decode_b32_h32_nk32768(cuda_lib):
    """The bench decode workload: B32 H32 Nq1 Nk32768 d128 bf16, 64 chunks of 512, 5% of the
    sequences truncated.  Inputs drawn on the device (17 GB); sampled (b, h) rows vs the oracle."""
    B, H, Nk, d = 32, 32, 32768, 128
    q, k, v = si.attn_inputs(B, H, 1, Nk, d, torch.bfloat16, seed=0, device="cuda")
    kv_len = si.decode_kv_len(B, Nk, seed=0)
    o, lse = cuda_lib.attn_splitkv(q, k, v, 64, kv_len=kv_len.cuda())
    torch.cuda.synchronize()
    cuda_lib.sync_status()
    trunc = torch.nonzero(kv_len < Nk).reshape(-1).tolist()
    picks = sorted(set([0, B - 1] + trunc + list(range(1, B, 7))))
    for b in picks:
        for h in (0, 17, H - 1):
            n = int(kv_len[b])
            ro, rl = oracle.attention(bf16_bits(q[b:b + 1, h:h + 1]), bf16_bits(k[b:b + 1, h:h + 1, :n]),
                                      bf16_bits(v[b:b + 1, h:h + 1, :n]))
            assert_lse_close(lse[b, h], rl)
            assert_out_close(o[b, h], ro[0, 0], BF16_O_ATOL)
    assert not torch.isnan(o).any()


@pytest.mark.parametrize("fill", [0x00, 0xFF, 0x01])
@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 2)])
def test_workspace_contents_do_not_matter(cuda_lib, fill, H, Hkv):
    # The workspace's contents on entry do not matter: every partial the merge reads is written by
    # the same call (an empty chunk writes O_c = 0, lse_c = -inf), whatever the workspace held
    # before (zeros, all ones, small values) and across repeated calls on the same workspace.
    # Grouped heads with two queries per row take the group kernel.
    oa = cuda_lib
    B, Nq, Nk, d, splits = 3, 2, 2000, 128, 16
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, Nq, Nk, d, torch.bfloat16, seed=fill + H)
    kv_len = [2000, 700, 0]
    kvd = torch.tensor(kv_len, dtype=torch.int32).cuda()
    ws = torch.full((oa.splitkv_workspace_bytes(B, H, Nq, d, splits),), fill, dtype=torch.uint8, device="cuda")
    g = H // Hkv
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k.repeat_interleave(g, dim=1)),
                              bf16_bits(v.repeat_interleave(g, dim=1)), kv_len=kv_len)
    out = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    for _ in range(3):
        out.fill_(7.0)
        lse.fill_(7.0)
        oa.attn_splitkv(q.cuda(), k.cuda(), v.cuda(), splits, kv_len=kvd, out=out, lse=lse, workspace=ws)
        torch.cuda.synchronize()
        oa.sync_status()
        assert_lse_close(lse, rl)
        assert_out_close(out, ro, BF16_O_ATOL, lse_ref=rl)
