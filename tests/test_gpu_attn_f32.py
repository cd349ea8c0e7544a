"""fp32 SIMT attention kernel (runtime Br/Bc tiles) vs the fp64 oracle (gpu)."""
import json
import math
import os

import pytest
import torch

import oracle
import synth_inputs as si
from parity import F32_ATTN_ATOL, assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _check(oa, q, k, v, causal=False, kv_len=None, tiles=None, atol=F32_ATTN_ATOL):
    kvd = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32).cuda()
    if tiles is None:
        o, lse = oa.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, kv_len=kvd)
    else:
        o, lse = oa.attn_fwd_f32_tiles(q.cuda(), k.cuda(), v.cuda(), tiles[0], tiles[1], causal=causal, kv_len=kvd)
    torch.cuda.synchronize()
    oa.sync_status()
    ro, rl = oracle.attention(q.numpy(), k.numpy(), v.numpy(), causal=causal, kv_len=kv_len)
    assert_lse_close(lse, rl)
    return assert_out_close(o, ro, atol, lse_ref=rl)


def test_lesson_worked_shapes_br4_bc3(cuda_lib):
    """Tiny fp32 config: Q, K, V [6, 4], Br = 4, Bc = 3, scale 1/2, non-causal."""
    ws = json.load(open(os.path.join(GOLD, "lesson_step2_shapes.json")))["walk_shapes"]
    q, k, v = si.attn_inputs(1, 1, ws["N"], ws["Nk"], ws["d"], torch.float32, seed=0)
    _check(cuda_lib, q, k, v, tiles=(ws["Br"], ws["Bc"]))


@pytest.mark.parametrize("N,Nk,d", json.load(open(os.path.join(GOLD, "lesson_step2_shapes.json")))["cases"])
def test_lesson_step2_cases(cuda_lib, N, Nk, d):
    q, k, v = si.attn_inputs(1, 1, N, Nk, d, torch.float32, seed=N + Nk)
    _check(cuda_lib, q, k, v, tiles=(4, 3))
    _check(cuda_lib, q, k, v)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tiles", [None, (1, 1), (4, 3), (16, 64), (64, 7)])
def test_masks_and_tiles(cuda_lib, causal, tiles):
    B, H, N, d = 3, 2, 77, 24
    q, k, v = si.attn_inputs(B, H, N, N, d, torch.float32, seed=5)
    _check(cuda_lib, q, k, v, causal=causal, kv_len=[77, 13, 0], tiles=tiles, atol=2e-5)


@pytest.mark.parametrize("d", [1, 4, 33, 128, 256])
def test_head_dims(cuda_lib, d):
    q, k, v = si.attn_inputs(2, 2, 40, 70, d, torch.float32, seed=d)
    _check(cuda_lib, q, k, v, atol=2e-5)


def test_closed_form_causal_row0_and_uniform_keys(cuda_lib):
    B, H, N, d = 1, 2, 50, 16
    q, k, v = si.attn_inputs(B, H, N, N, d, torch.float32, seed=9)
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0])  # row 0 sees only key 0: exactly V_0
    kz = torch.zeros_like(k)
    o, lse = cuda_lib.attn_fwd(q.cuda(), kz.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert torch.allclose(o.cpu(), v.mean(2, keepdim=True).expand_as(o), atol=1e-6)
    assert torch.allclose(lse.cpu(), torch.full_like(lse.cpu(), math.log(N)), atol=1e-6)
