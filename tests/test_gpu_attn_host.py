"""GPU tests of the host-buffer forward (oa_attn_fwd_host): copies in, kernels and copies out of
pieces of the key/value head planes overlapped on the library's streams.  Every piece runs the same
kernel as oa_attn_fwd_gqa on its heads, so the outputs must equal attn_fwd's bit for bit; one case
is also checked against the fp64 oracle with the forward's tolerances."""
import numpy as np
import pytest
import torch

import online_softmax_attention_tiled_gb300 as oa
import oracle
import synth_inputs as si
from parity import BF16_O_ATOL, LSE_ATOL, assert_lse_close, bf16_bits, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _pinned(*ts):
    return [t.contiguous().pin_memory() for t in ts]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal,chunks", [
    (1, 4, 4, 300, 128, True, 0),
    (2, 8, 2, 257, 64, False, 3),
    (1, 3, 3, 129, 128, True, 64),   # more pieces requested than planes
    (1, 2, 1, 200, 128, True, 1),    # one piece: no overlap, same result
    (3, 4, 4, 64, 64, False, 5),
    # several rounds of the persistent grid (odd rounds read key tiles top down) and, with 64 MiB of
    # K/V, two phases over bands of heads: each piece must follow the whole call's order
    (1, 16, 16, 4096, 128, True, 3),
    (1, 32, 16, 8192, 128, True, 3),
])
def test_host_forward_equals_device_forward(B, H, Hkv, N, d, causal, chunks):
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, N, N, d, torch.bfloat16, seed=11 + N)
    qh, kh, vh = _pinned(q, k, v)
    o, lse = oa.attn_fwd_host(qh, kh, vh, causal=causal, chunks=chunks)
    torch.cuda.synchronize()
    ro, rl = oa.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o, ro.cpu())
    assert torch.equal(lse, rl.cpu())


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,chunks", [
    (1, 32, 8, 1024, 16384, 3),   # 64 MiB of K/V, items of near-equal weight: dealt plane by plane
    (1, 16, 16, 2048, 8192, 4),   # 64 MiB of K/V, items of unequal weight: dealt in phases
])
def test_host_forward_with_a_key_offset_equals_device_forward(B, H, Hkv, Nq, Nk, chunks):
    # new queries after a cache, cut into pieces: each piece must sum its key tiles in the order
    # of the whole call (bottom up throughout when the call is dealt plane by plane)
    q, k, v = si.attn_inputs_gqa(B, H, Hkv, Nq, Nk, 128, torch.bfloat16, seed=Nq + Nk)
    qh, kh, vh = _pinned(q, k, v)
    o, lse = oa.attn_fwd_host(qh, kh, vh, causal=True, chunks=chunks)
    torch.cuda.synchronize()
    ro, rl = oa.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, ro.cpu())
    assert torch.equal(lse, rl.cpu())


def test_host_forward_matches_oracle_and_skips_lse():
    q, k, v = si.attn_inputs(1, 2, 300, 300, 128, torch.bfloat16, seed=4)
    o, lse = oa.attn_fwd_host(*_pinned(q, k, v), causal=True, chunks=2)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(bf16_bits(q), bf16_bits(k), bf16_bits(v), causal=True)
    assert np.abs(to_np(o) - ro).max() <= BF16_O_ATOL
    assert_lse_close(lse, rl, LSE_ATOL)
    o2, lse2 = oa.attn_fwd_host(*_pinned(q, k, v), causal=True, want_lse=False)
    torch.cuda.synchronize()
    assert lse2 is None and torch.equal(o2, o)


def test_host_forward_fp32_and_back_to_back_calls():
    # fp32 runs the SIMT kernel per piece; two calls in a row reuse one workspace, and the second
    # call's copies must wait for the first call's kernels
    q, k, v = si.attn_inputs(2, 2, 40, 40, 32, torch.float32, seed=6)
    q2, k2, v2 = si.attn_inputs(2, 2, 40, 40, 32, torch.float32, seed=9)
    ws = torch.empty(oa.attn_fwd_host_workspace_bytes(torch.float32, 2, 2, 2, 40, 40, 32), dtype=torch.uint8,
                     device=DEV)
    o1, l1 = oa.attn_fwd_host(*_pinned(q, k, v), chunks=4, workspace=ws)
    o2, l2 = oa.attn_fwd_host(*_pinned(q2, k2, v2), chunks=4, workspace=ws)
    torch.cuda.synchronize()
    r1, rl1 = oa.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV))
    r2, rl2 = oa.attn_fwd(q2.to(DEV), k2.to(DEV), v2.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(o1, r1.cpu()) and torch.equal(l1, rl1.cpu())
    assert torch.equal(o2, r2.cpu()) and torch.equal(l2, rl2.cpu())


def test_host_forward_rejects_device_tensors():
    q, k, v = si.attn_inputs(1, 1, 8, 8, 64, torch.bfloat16, seed=1)
    with pytest.raises(oa.OAError):
        oa.attn_fwd_host(q.to(DEV), k, v)
