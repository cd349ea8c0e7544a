"""Runs one kernel case a few times on cuda:0, for use under a profiler.

  python -m online_softmax_attention_tiled_gb300.profile_case CASE [--reps R] [--batch B]

Cases (inputs seeded as in the benchmark):
  attn_causal      causal attention fwd bf16, B=1 H=32 N=8192 d=128 (~256 MiB on the device)
  attn_noncausal   non-causal attention fwd bf16, B=4 H=16 N=4096 d=64
  attn_bwd_causal  causal attention bwd bf16, B=1 H=32 N=8192 d=128 (O and LSE from the forward;
                   ~650 MiB on the device)
  attn_varlen      causal attention fwd bf16 over 16 packed sequences of 1024-8192 tokens (96634 in
                   all), H=32 H_kv=8 d=128 (~1 GiB on the device)
  softmax          row softmax + LSE fp32 [4096, 32768] (1 GiB)
  decode           split-KV decode bf16, B (default 4) x H=32, Nk=32768, d=128, 64 chunks
                   (--batch 32 is the full 17 GB benchmark shape)
  decode_gqa       decode bf16 over a grouped cache, B (default 4) x H=32, H_kv=8, Nk=32768, d=128,
                   each group's queries as rows of the tensor-core forward (--batch 32: 4.3 GB)
Prints the mean CUDA-event time per launch.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import online_softmax_attention_tiled_gb300 as oa  # noqa: E402
import synth_inputs as si  # noqa: E402


def make_case(name, dev, batch):
    if name == "attn_causal":
        q, k, v = si.attn_inputs(1, 32, 8192, 8192, 128, torch.bfloat16, seed=0, device=dev)
        o, lse = torch.empty_like(q), torch.empty((1, 32, 8192), device=dev)
        return lambda: oa.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
    if name == "attn_noncausal":
        q, k, v = si.attn_inputs(4, 16, 4096, 4096, 64, torch.bfloat16, seed=0, device=dev)
        o, lse = torch.empty_like(q), torch.empty((4, 16, 4096), device=dev)
        return lambda: oa.attn_fwd(q, k, v, out=o, lse=lse)
    if name == "attn_bwd_causal":
        q, k, v = si.attn_inputs(1, 32, 8192, 8192, 128, torch.bfloat16, seed=0, device=dev)
        do = si.randn((1, 32, 8192, 128), 3, torch.bfloat16, dev)
        o, lse = oa.attn_fwd(q, k, v, causal=True)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(oa.attn_bwd_workspace_bytes(1, 32, 8192, 128), dtype=torch.uint8, device=dev)
        return lambda: oa.attn_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
    if name == "attn_varlen":
        lens = si.varlen_lengths(16, 8192, seed=0, min_len=1024)
        q, k, v, cq, ck = si.varlen_inputs(lens, lens, 32, 8, 128, torch.bfloat16, seed=0, device=dev)
        cq, ck = cq.to(dev), ck.to(dev)
        mx = int(max(lens))
        o, lse = torch.empty_like(q), torch.empty((q.shape[0], 32), device=dev)
        return lambda: oa.attn_fwd_varlen(q, k, v, cq, ck, mx, mx, causal=True, out=o, lse=lse)
    if name == "softmax":
        x, *_ = si.softmax_input(4096, 32768, seed=0)
        x = x.to(dev)
        y, lse = torch.empty_like(x), torch.empty(4096, device=dev)
        return lambda: oa.softmax_rows(x, y=y, lse=lse)
    if name == "decode":
        q, k, v = si.attn_inputs(batch, 32, 1, 32768, 128, torch.bfloat16, seed=0, device=dev)
        kv = si.decode_kv_len(batch, 32768, seed=0).to(dev)
        o, lse = torch.empty_like(q), torch.empty((batch, 32, 1), device=dev)
        ws = torch.empty(oa.splitkv_workspace_bytes(batch, 32, 1, 128, 64), dtype=torch.uint8, device=dev)
        return lambda: oa.attn_splitkv(q, k, v, 64, kv_len=kv, out=o, lse=lse, workspace=ws)
    if name == "decode_gqa":
        q, k, v = si.attn_inputs_gqa(batch, 32, 8, 1, 32768, 128, torch.bfloat16, seed=0, device=dev)
        kv = si.decode_kv_len(batch, 32768, seed=0).to(dev)
        o, lse = torch.empty_like(q), torch.empty((batch, 32, 1), device=dev)
        ws = torch.empty(oa.splitkv_workspace_bytes(batch, 32, 1, 128, 64), dtype=torch.uint8, device=dev)
        return lambda: oa.attn_splitkv(q, k, v, 64, kv_len=kv, out=o, lse=lse, workspace=ws)
    raise SystemExit(f"unknown case {name}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--batch", type=int, default=4)
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fn = make_case(a.case, dev, a.batch)
    fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(a.reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    oa.sync_status()
    print(f"{a.case}: {sum(times) / len(times):.4f} ms per launch over {a.reps} launches")


if __name__ == "__main__":
    main()
