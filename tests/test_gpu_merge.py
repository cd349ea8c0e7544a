"""LSE merge kernel vs the fp64 oracle merge (gpu)."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_lse_close, assert_out_close, to_np

pytestmark = pytest.mark.gpu
NEG_INF = float("-inf")


def _partials(S, R, d, seed, frac_empty=0.2):
    g = torch.Generator().manual_seed(seed)
    po = torch.randn(S, R, d, generator=g) if d > 0 else None
    pl = torch.randn(S, R, generator=g) * 3 + 5
    pl[torch.rand(S, R, generator=g) < frac_empty] = NEG_INF
    pl[:, 0] = NEG_INF  # a row with no visible key at all
    if po is not None:
        po[torch.isneginf(pl)] = 0.0  # empty partials carry o_c = 0
    return po, pl


@pytest.mark.parametrize("S,R,d", [(1, 5, 8), (5, 37, 0), (5, 37, 7), (64, 1024, 128), (3, 100, 64), (17, 9, 1024)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_merge_vs_oracle(cuda_lib, S, R, d, out_dtype):
    po, pl = _partials(S, R, d, seed=S * 1000 + R + d)
    ro, rl = oracle.lse_merge(None if po is None else po.double().numpy(), pl.double().numpy())
    o, lse = cuda_lib.lse_merge(None if po is None else po.cuda(), pl.cuda(), out_dtype=out_dtype)
    torch.cuda.synchronize()
    cuda_lib.sync_status()
    assert_lse_close(lse, rl)
    if d > 0:
        atol = 2e-2 if out_dtype == torch.bfloat16 else 2e-6
        assert_out_close(o, ro, atol, lse_ref=rl)


def test_merge_is_order_free(cuda_lib):
    po, pl = _partials(9, 64, 32, seed=3)
    perm = torch.randperm(9, generator=torch.Generator().manual_seed(1))
    o1, l1 = cuda_lib.lse_merge(po.cuda(), pl.cuda())
    o2, l2 = cuda_lib.lse_merge(po[perm].contiguous().cuda(), pl[perm].contiguous().cuda())
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_np(o1), to_np(o2), rtol=0, atol=1e-6)
    assert_lse_close(l2, to_np(l1), atol=1e-6)
