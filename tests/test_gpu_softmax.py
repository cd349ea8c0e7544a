"""Row softmax + LSE kernel vs the fp64 oracle (gpu)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from parity import assert_lse_close, assert_softmax_close, to_np

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _run(oa, x, **kw):
    y, lse = oa.softmax_rows(x.cuda(), **kw)
    torch.cuda.synchronize()
    oa.sync_status()
    return y, lse


def test_worked_examples(cuda_lib):
    oa = cuda_lib
    g = json.load(open(os.path.join(GOLD, "roadmap_s3_worked_example.json")))
    y, lse = _run(oa, torch.tensor([g["x"]], dtype=torch.float32))
    assert np.all(np.abs(to_np(y)[0] - np.array(g["y"])) <= 0.5e-4)
    ry, rl = oracle.softmax_rows(np.array([g["x"]], np.float32))
    assert_softmax_close(y, ry)
    assert_lse_close(lse, rl)
    g = json.load(open(os.path.join(GOLD, "lesson_step1_stats.json")))
    y, lse = _run(oa, torch.tensor([g["x"]], dtype=torch.float32))
    ry, rl = oracle.softmax_rows(np.array([g["x"]], np.float32))
    assert_softmax_close(y, ry)
    assert_lse_close(lse, rl)
    assert abs(float(lse[0]) - (g["m"] + np.log(g["l"]))) < 1e-4


@pytest.mark.parametrize("cols", [1, 3, 37, 128, 1000, 1023, 1025, 2048, 4097, 8192, 8193, 20000, 32768, 40960,
                                  40964, 65536, 70001, 98304, 131072, 131073, 200003, 262144, 262148, 400000])
def test_ragged_widths_with_masks(cuda_lib, cols):
    rows = 24
    x, full, pre, _ = si.softmax_input(rows, cols, seed=cols, frac_full=0.1, frac_prefix=0.3)
    y, lse = _run(cuda_lib, x)
    ry, rl = oracle.softmax_rows(x.numpy())
    assert_softmax_close(y, ry)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("cols", [70001, 150001, 262145])
def test_wide_unaligned_rows(cuda_lib, cols):
    # odd widths: rows are not 16-byte aligned, so the scalar form of the wide instance runs (one read
    # up to 16 x 16384 columns, streaming beyond)
    x, *_ = si.softmax_input(6, cols, seed=cols + 1, frac_full=0.2, frac_prefix=0.4)
    y, lse = _run(cuda_lib, x)
    ry, rl = oracle.softmax_rows(x.numpy())
    assert_softmax_close(y, ry)
    assert_lse_close(lse, rl)


def test_unaligned_rows_and_strided_slices_lesson_chunks(cuda_lib):
    """The lesson's [8, 37] matrix, its column chunks [5,1,13,8,10] run as strided
    slices (row stride 37: scalar path), then merged by LSE on the GPU."""
    oa = cuda_lib
    X = si.lesson_matrix(seed=0)
    Xd = X.cuda()
    _, full_lse_ref = oracle.softmax_rows(X.numpy())
    parts, c0 = [], 0
    for w in si.LESSON_CHUNKS:
        sl = Xd[:, c0:c0 + w]
        y, lse = oa.softmax_rows(sl)
        ry, rl = oracle.softmax_rows(X[:, c0:c0 + w].numpy())
        assert_softmax_close(y, ry, what=f"chunk at {c0}")
        assert_lse_close(lse, rl, what=f"chunk lse at {c0}")
        parts.append(lse)
        c0 += w
    part_lse = torch.stack(parts).contiguous()
    _, merged = oa.lse_merge(None, part_lse)
    torch.cuda.synchronize()
    assert_lse_close(merged, full_lse_ref, what="merged lse")
    assert float(merged[2]) == float("-inf")


@pytest.mark.parametrize("cols", [3000, 16384])
def test_in_place_and_outputs_optional(cuda_lib, cols):
    oa = cuda_lib
    x, *_ = si.softmax_input(16, cols, seed=4)
    ry, rl = oracle.softmax_rows(x.numpy())
    xd = x.cuda()
    y, lse = oa.softmax_rows(xd, y=xd)  # in place
    torch.cuda.synchronize()
    assert y.data_ptr() == xd.data_ptr()
    assert_softmax_close(xd, ry)
    assert_lse_close(lse, rl)
    y, lse = oa.softmax_rows(x.cuda(), want_y=False)
    assert y is None
    assert_lse_close(lse, rl)
    y, lse = oa.softmax_rows(x.cuda(), want_lse=False)
    assert lse is None
    assert_softmax_close(y, ry)


def test_fp32_overflow_argument(cuda_lib):
    y, lse = _run(cuda_lib, torch.tensor([[89.0, 0.0], [-1e30, 0.0]], dtype=torch.float32))
    ry, rl = oracle.softmax_rows(np.array([[89.0, 0.0], [-1e30, 0.0]], np.float32))
    assert_softmax_close(y, ry)
    assert_lse_close(lse, rl)


@pytest.mark.slow
def test_full_size_4096x32768(cuda_lib):
    """The bench workload: 4096 x 32768 fp32, N(0,1)*4, 1% rows fully -inf, 10% -inf prefixes.
    Compared on a sampled row set that includes every fully masked row and 64 prefix rows."""
    x, full, pre, _ = si.softmax_input(4096, 32768, seed=0)
    y, lse = _run(cuda_lib, x)
    rows = torch.unique(torch.cat([si.sample_rows(4096, 192, seed=1), full, pre[:64]])).numpy()
    ry, rl = oracle.softmax_rows(x[rows].numpy())
    assert_softmax_close(y[torch.from_numpy(rows).cuda()], ry)
    assert_lse_close(lse[torch.from_numpy(rows).cuda()], rl)
    # properties that hold on every row: fully masked rows are all zero, -inf elements give +0.0, rows sum to 1
    assert torch.all(y[full.cuda()] == 0)
    assert torch.all(torch.isneginf(lse[full.cuda()]))
    assert not torch.isnan(y).any()
    xm = torch.isneginf(x.cuda())
    assert torch.all(y[xm] == 0)
    live = ~torch.isneginf(lse)
    s = y[live].double().sum(1)
    assert torch.allclose(s, torch.ones_like(s), atol=1e-5)
