"""bf16 tensor-core attention kernel (tcgen05 / TMEM / TMA) vs the fp64 oracle (gpu)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import BF16_O_ATOL, assert_lse_close, assert_out_close, bf16_bits

pytestmark = pytest.mark.gpu


def _run(oa, q, k, v, causal=False, kv_len=None, scale=None):
    kvd = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32).cuda()
    o, lse = oa.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, kv_len=kvd, scale=scale)
    torch.cuda.synchronize()
    oa.sync_status()
    return o, lse


def _check(oa, q, k, v, causal=False, kv_len=None, scale=None, lse_atol=None):
    o, lse = _run(oa, q, k, v, causal, kv_len, scale)
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=causal, kv_len=kv_len,
                              scale=scale)
    if lse_atol is None:
        assert_lse_close(lse, rl)
    else:
        assert_lse_close(lse, rl, atol=lse_atol)
    return assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)


@pytest.mark.parametrize("d", [64, 128])
def test_single_tile(cuda_lib, d):
    q, k, v = si.attn_inputs(1, 1, 128, 128, d, torch.bfloat16, seed=d)
    _check(cuda_lib, q, k, v)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 129, 256, 300, 640])
def test_square_ragged(cuda_lib, d, causal, N):
    q, k, v = si.attn_inputs(2, 3, N, N, d, torch.bfloat16, seed=N * 7 + d)
    _check(cuda_lib, q, k, v, causal=causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(200, 333), (513, 64), (1, 1000), (256, 1)])
def test_rectangular_noncausal(cuda_lib, d, Nq, Nk):
    q, k, v = si.attn_inputs(2, 2, Nq, Nk, d, torch.bfloat16, seed=Nq + Nk)
    _check(cuda_lib, q, k, v)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_kv_len_masks(cuda_lib, d, causal):
    N = 384
    q, k, v = si.attn_inputs(4, 2, N, N, d, torch.bfloat16, seed=11)
    _check(cuda_lib, q, k, v, causal=causal, kv_len=[N, 1, 0, 200])



@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(64, 300), (128, 1), (3, 129), (100, 1000), (128, 640)])
def test_short_query_block_splits_keys_between_slots(cuda_lib, d, Nq, Nk):
    # At most 128 query rows without the mask: both query-tile slots take the same rows
    # over alternate key tiles, each with its own running max, sum and O, merged per row at the
    # end.  Odd and even numbers of key tiles, a slot with no tile at all (one key tile), a batch
    # entry with no keys, a ragged key end, and large scores (each slot rescales on its own).
    q, k, v = si.attn_inputs(2, 3, Nq, Nk, d, torch.bfloat16, seed=5 * Nq + Nk + d)
    _check(cuda_lib, q, k, v)
    _check(cuda_lib, q, k, v, kv_len=[Nk // 2 + 1, 0])
    _check(cuda_lib, q, k, v, scale=1.0)


@pytest.mark.parametrize("d", [64, 128])
def test_output_16_byte_aligned(cuda_lib, d):
    # O rows are written with 32-byte stores when o is 32-byte aligned; an o that is only
    # 16-byte aligned (the documented minimum) takes the 16-byte store path.
    B, H, N = 1, 3, 300
    q, k, v = si.attn_inputs(B, H, N, N, d, torch.bfloat16, seed=31 + d)
    flat = torch.empty(B * H * N * d + 8, dtype=torch.bfloat16, device="cuda")
    out = flat[8:].view(B, H, N, d)  # 16 bytes past a 256-byte aligned allocation
    assert out.data_ptr() % 32 == 16
    o, lse = cuda_lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, out=out)
    torch.cuda.synchronize()
    cuda_lib.sync_status()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True)
    assert_lse_close(lse, rl)
    assert_out_close(o, ro, BF16_O_ATOL, lse_ref=rl)

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_many_items_per_cta(cuda_lib, d, causal):
    # B*H = 160 heads x 3 query blocks = 480 work items: more than one SM's worth each, so
    # every CTA of the persistent grid runs several items in turn.  The last query block's
    # second tile lies past Nq, one sequence has no keys at all (an item with no work
    # between items with work) and the others end mid-tile.
    N = 640
    q, k, v = si.attn_inputs(4, 40, N, N, d, torch.bfloat16, seed=21 + d)
    _check(cuda_lib, q, k, v, causal=causal, kv_len=[N, 0, 129, 511])


def test_scale_and_large_scores(cuda_lib):
    q, k, v = si.attn_inputs(1, 2, 300, 300, 128, torch.bfloat16, seed=12)
    _check(cuda_lib, q, k, v, scale=1.0)  # scores ~N(0, 128): exercises large max shifts
    _check(cuda_lib, q, k, v, scale=0.01)
    # Scaled scores spread over hundreds of log2 units: most exponentials
    # underflow to +0 and rows rescale often.  Here LSE ~ max_j s_j * scale ~ 300,
    # and it inherits the fp32 accumulation error of the score itself: about
    # sqrt(d) * 2^-24 * sum_i |q_i k_i| per score, times the scale.  The flat 1e-4
    # bound is for scale = 1/sqrt(d); at scale 8 the bound is that product.
    qf, kf = q.float().numpy(), k.float().numpy()
    abs_dot = np.einsum("bhqd,bhkd->bhqk", np.abs(qf), np.abs(kf)).max()
    lse_atol = 1e-4 + 8.0 * 4 * math.sqrt(128) * 2.0 ** -24 * abs_dot
    _check(cuda_lib, q, k, v, scale=8.0, lse_atol=lse_atol)
    _check(cuda_lib, q, k, v, causal=True, scale=8.0, lse_atol=lse_atol)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_running_max_grows_every_key_tile(cuda_lib, d, causal):
    # Scores that climb ~40 log2 units per 128-key tile for even query rows and fall for odd ones:
    # every key tile raises the running max of half the lanes of every warp past the lazy-rescale
    # threshold (O and l rescaled before the next PV), and leaves the other half's untouched.
    B, H, N = 1, 2, 512
    sign = torch.ones(N, dtype=torch.float32)
    sign[1::2] = -1.0
    q = sign.view(1, 1, N, 1).expand(B, H, N, d).contiguous()
    ramp = 0.02 * torch.arange(N, dtype=torch.float32).view(1, 1, N, 1)
    k = ramp + 0.05 * si.randn((B, H, N, d), 31, torch.float32)
    v = si.randn((B, H, N, d), 32, torch.float32)
    q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    qf, kf = q.float().numpy(), k.float().numpy()
    abs_dot = np.einsum("bhqd,bhkd->bhqk", np.abs(qf), np.abs(kf)).max()
    lse_atol = 1e-4 + 4 * math.sqrt(d) * 2.0 ** -24 * abs_dot / math.sqrt(d)
    _check(cuda_lib, q, k, v, causal=causal, lse_atol=lse_atol)


def test_causal_row0_closed_form(cuda_lib):
    q, k, v = si.attn_inputs(1, 4, 256, 256, 128, torch.bfloat16, seed=13)
    o, lse = _run(cuda_lib, q, k, v, causal=True)
    assert torch.allclose(o[:, :, 0].float().cpu(), v[:, :, 0].float(), atol=1e-2)
    ref = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1) / math.sqrt(128)
    assert torch.allclose(lse[:, :, 0].double().cpu(), ref, atol=1e-4)


def _sampled_full_size(oa, B, H, N, d, causal, seed, per_head):
    q, k, v = si.attn_inputs(B, H, N, N, d, torch.bfloat16, seed=seed)
    o, lse = _run(oa, q, k, v, causal=causal)
    local = si.sample_rows(N, per_head, seed=seed)
    rows = (torch.arange(B * H)[:, None] * N + local[None, :]).reshape(-1).numpy()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=causal, rows=rows)
    og = o.reshape(-1, d)[torch.from_numpy(rows).cuda()]
    lg = lse.reshape(-1)[torch.from_numpy(rows).cuda()]
    assert_lse_close(lg, rl)
    err = assert_out_close(og, ro, BF16_O_ATOL)
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    return err


@pytest.mark.slow
def test_full_size_noncausal_b4_h16_n4096_d64(cuda_lib):
    _sampled_full_size(cuda_lib, 4, 16, 4096, 64, False, seed=0, per_head=96)


@pytest.mark.slow
def test_full_size_causal_b1_h32_n8192_d128(cuda_lib):
    _sampled_full_size(cuda_lib, 1, 32, 8192, 128, True, seed=0, per_head=160)
