"""The debug build (OA_DEBUG=1 loads liboa_debug.so: the kernels check the bounds and alignment of
their computed global accesses and record a failed check in the status word) against the release
library (gpu).  Small and odd shapes run through every checked kernel -- the row softmax (one CTA,
clusters with the serial and the parallel merge, the unaligned scalar path), the tensor-core
forward (both head sizes, square and offset causal, grouped heads, packed sequences) and both
backward kernels -- in two subprocesses, one per build: no check fires (sync_status is OK) and
every output is bit-identical (but the backward's dQ, summed by fp32 reduce-adds in arrival order,
which may differ by a rounding), so the checks change nothing but the reporting.  A check that fails
on purpose (oa_selftest_debug_check) is reported as OA_ERR_INVALID, its store skipped, by the debug
build alone.
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys, torch
sys.path.insert(0, sys.argv[2])
import online_softmax_attention_tiled_gb300 as oa
import synth_inputs as si
assert oa.DEBUG == (sys.argv[3] == "1"), "wrong library loaded"
dev = "cuda"
out = {}
for rows, cols in ((37, 1), (5, 6), (3, 129), (4, 4099), (2, 40003), (3, 70001), (2, 131072)):
    x = si.softmax_input(rows, cols, seed=cols)[0].to(dev)
    y, l = oa.softmax_rows(x)
    out["softmax %dx%d" % (rows, cols)] = (y, l)
x = si.softmax_input(3, 5001, seed=5)[0].to(dev)
xs = torch.empty(3, 5003, device=dev)[:, 1:5002]  # unaligned rows: the scalar path
xs.copy_(x)
out["softmax unaligned"] = oa.softmax_rows(xs)
for d in (64, 128):
    for nq, nk, causal in ((1, 1, False), (6, 37, True), (37, 6, True), (129, 129, True), (300, 517, False), (257, 600, True)):
        q, k, v = si.attn_inputs(2, 2, nq, nk, d, torch.bfloat16, seed=7 * nq + nk + d)
        out["fwd d%d %d %d %d" % (d, nq, nk, causal)] = oa.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    q, k, v = si.attn_inputs_gqa(2, 8, 2, 3, 700, d, torch.bfloat16, seed=d)
    out["fwd gqa decode d%d" % d] = oa.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
    lq, lk = [5, 130, 1, 0], [40, 130, 7, 9]
    q, k, v, cq, ck = si.varlen_inputs(lq, lk, 4, 2, d, torch.bfloat16, seed=d + 1)
    out["fwd varlen d%d" % d] = oa.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev),
                                                   max(lq), max(lk), causal=True)
    q, k, v = si.attn_inputs(1, 2, 200, 333, d, torch.bfloat16, seed=d + 2)
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    o, lse = oa.attn_fwd(q, k, v, causal=True)
    do = si.randn((1, 2, 200, d), d + 3, torch.bfloat16, dev)
    out["bwd d%d" % d] = oa.attn_bwd(q, k, v, o, lse, do, causal=True)
oa.sync_status()  # raises if a check fired
torch.save({key: tuple(t.cpu() for t in val) for key, val in out.items()}, sys.argv[1])
# a check that fails on purpose: reported (and its store skipped) only by the debug build
flag = oa.selftest_debug_check()
try:
    oa.sync_status()
    reported = False
except oa.OAError as e:
    reported = e.status == oa.OA_ERR_INVALID
print("check", flag, int(reported))
oa.sync_status()  # the word was cleared: later calls start clean
print("ok", len(out))
'''


def _run(tmp_path, debug: bool):
    script = tmp_path / "run_builds.py"
    script.write_text(SCRIPT)
    dest = tmp_path / ("debug.pt" if debug else "release.pt")
    env = dict(os.environ)
    env["OA_DEBUG"] = "1" if debug else "0"
    r = subprocess.run([sys.executable, str(script), str(dest), ROOT, "1" if debug else "0"], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    check = [ln for ln in r.stdout.splitlines() if ln.startswith("check ")]
    assert check == (["check 0 1"] if debug else ["check 1 0"]), r.stdout[-2000:]
    return torch.load(dest)


def _bits(t):
    """The tensor's bit pattern (so that -0.0, +0.0 and -inf compare exactly)."""
    return t.contiguous().view(torch.uint8)


def test_debug_build_matches_release_and_no_check_fires(tmp_path):
    rel = _run(tmp_path, debug=False)
    dbg = _run(tmp_path, debug=True)
    assert rel.keys() == dbg.keys()
    for key in rel:
        assert len(rel[key]) == len(dbg[key]), key
        for i, (a, b) in enumerate(zip(rel[key], dbg[key])):
            assert a.dtype == b.dtype and a.shape == b.shape, key
            if key.startswith("bwd") and i == 0:
                # dQ: the same fp32 terms added in arrival order, then rounded to bf16 -- equal up to
                # one bf16 rounding of the sum
                assert torch.allclose(a.float(), b.float(), rtol=2.0 ** -7, atol=1e-6), key
            else:
                assert torch.equal(_bits(a), _bits(b)), key
