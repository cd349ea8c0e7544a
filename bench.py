"""Benchmark of the online-softmax tiled attention library on GB300.

Prints ONE JSON line (rank 0).  The headline workload is the fused causal
attention forward, bf16, B=1 H=32 N=8192 d=128 (one "step" = one forward
over that batch).  The other hot-path kernels (the row softmax + LSE on fp32
[4096, 32768] -- the metric's second half --, the non-causal B4 H16 N4096 d64
forward, split-KV decode, decode over a grouped cache, a causal forward over
packed sequences, the backward passes) are measured in the same run and
reported under "components", each against its own roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--components/--no-components] [--no-cpu-baseline]
                  [--min-seconds S]
  python bench.py --case NAME [--reps R] [--batch B]     (one case, for a profiler)

Timing: W untimed warm-up steps, then the K-step loop is repeated until the
timed region lasts at least --min-seconds (default 3 s), so that the clock
record describes it; per-step figures come from every timed step.  Each
launch is bracketed by CUDA events on the launching stream.

--impl reference times the CPU oracle (the only reference this method has:
the pages carry no implementation) on a bounded sample of the same workload.
For N > 1 (torchrun) every rank runs its own replica of the workload on its
own GPU (independent batches, no collective on the data path); timing is the
max over ranks and "value" counts the work of all ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s (bf16, causal N=8192 d=128) & % tensor peak; softmax GB/s % HBM"
WORKLOAD = "causal attention fwd bf16 B=1 H=32 Nq=Nk=8192 d=128 scale=1/sqrt(128)"
B, H, N, D = 1, 32, 8192, 128
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Dense bf16 tensor work one SM retires per clock: one 128 x 128 x 16 MMA (524,288 FLOPs) per
# 64 cycles.  x SM count x SM clock = the hardware peak at the clock actually seen.
BF16_FLOP_PER_SM_CLOCK = 8192


# --------------------------------------------------------------------------
# work accounting (algorithmic, per launch)
# --------------------------------------------------------------------------
def causal_attn_flops(b, h, n, d):
    """4*d FLOPs (QK^T and PV) per visible (query, key) pair; n(n+1)/2 pairs per head."""
    return 4.0 * b * h * d * n * (n + 1) / 2


def dense_attn_flops(b, h, nq, nk, d):
    return 4.0 * b * h * nq * nk * d


def causal_pairs(nq, nk):
    """Visible (query, key) pairs of one head when query i sees keys j <= i + (nk - nq)."""
    off = nk - nq
    return sum(max(0, min(nk, i + off + 1)) for i in range(nq))


def kvcache_causal_flops(b, h, nq, nk, d):
    """4*d FLOPs per visible pair, the new queries being the last nq positions of nk keys."""
    return 4.0 * b * h * d * causal_pairs(nq, nk)


def causal_attn_bwd_flops(b, h, n, d):
    """10*d FLOPs per visible (query, key) pair: S = QK^T and dP = dO V^T recomputed, then dV, dK, dQ."""
    return 2.5 * causal_attn_flops(b, h, n, d)


def dense_attn_bwd_flops(b, h, nq, nk, d):
    return 2.5 * dense_attn_flops(b, h, nq, nk, d)


def softmax_bytes(rows, cols):
    """Read X once, write Y and LSE (fp32)."""
    return 4.0 * rows * cols * 2 + 4.0 * rows


def decode_bytes(b, h, d, kv_len_sum, esize=2, h_kv=None, nq=1):
    """q, the visible K and V rows (h_kv heads; default h), O and LSE, for nq new tokens per sequence."""
    h_kv = h if h_kv is None else h_kv
    return esize * (2.0 * h_kv * d * kv_len_sum + b * h * nq * d * 2) + 4.0 * b * h * nq


def varlen_causal_flops(lengths, h, d):
    """4*d FLOPs per visible (query, key) pair, L(L+1)/2 pairs per head of a sequence of length L."""
    return sum(4.0 * h * d * n * (n + 1) / 2 for n in lengths)


# --------------------------------------------------------------------------
# environment helpers
# --------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def code_digest(texts):
    """Digest of source texts with their // comments, trailing blanks and blank lines left out, so that
    an edit of the comments alone keeps a profile taken on the same code current."""
    h = hashlib.sha256()
    for text in texts:
        code = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(ln.rstrip() for ln in code.splitlines() if ln.strip()).encode())
    return h.hexdigest()[:16]


def kernel_source_digest():
    """code_digest of the attention kernel's sources."""
    texts = []
    for f in ("attn_tc.cu", "oa_common.cuh"):
        with open(os.path.join(ROOT, "online_softmax_attention_tiled_gb300", "csrc", f), encoding="utf-8") as fh:
            texts.append(fh.read())
    return code_digest(texts)


def profiled_traffic():
    """dram bytes per launch of the attention kernel from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "attn_fwd_tc_causal_b1h32n8192d128.md")
    try:
        text = open(p).read()
    except OSError:
        return None
    m_src = re.search(r"kernel_source_digest:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_src or not m_b or m_src.group(1) != kernel_source_digest():
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 20 ms while running.  Started before the
    warm-up; wait_first() blocks until nvidia-smi has produced a sample, so the timed region that
    follows is covered from its start."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.unparsed = 0
        self.error = None
        self.proc = None
        self.thread = None
        self._first = threading.Event()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
        except OSError as e:
            self.proc = None
            self.error = f"nvidia-smi not started: {e}"
            self._first.set()
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    @staticmethod
    def parse(line):
        """(sm MHz, max SM MHz, power W, {reason: active}) of one csv line, or None."""
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            return None
        try:
            sm, smax = float(parts[1]), float(parts[2])
        except ValueError:
            return None
        try:
            pw = float(parts[3])
        except ValueError:
            pw = float("nan")
        act = {n: v.lower().startswith("active") for n, v in zip(ClockSampler.REASONS, parts[5:9])}
        return sm, smax, pw, act

    def _read(self):
        for line in self.proc.stdout:
            r = self.parse(line)
            if r is None:
                self.unparsed += 1
                if self.unparsed == 1:
                    self.error = f"unparsed nvidia-smi line: {line.strip()[:160]}"
            else:
                self.samples.append((time.time(), r))
            self._first.set()
        self._first.set()

    def wait_first(self, timeout=10.0):
        self._first.wait(timeout)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if not self.samples and self.error is None:
                err = (self.proc.stderr.read() or "").strip() if self.proc.stderr else ""
                self.error = f"no samples; nvidia-smi said: {err[:200]}" if err else "no samples"
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [r for ts, r in self.samples if t0 <= ts <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "error": self.error or "no sample inside the timed region"}
        reasons = sorted({n for r in inside for n, a in r[3].items() if a})
        out = {"sm_mhz": statistics.median(r[0] for r in inside), "sm_max_mhz": max(r[1] for r in inside),
               "reasons": reasons, "samples": len(inside),
               "power_w_max": max((r[2] for r in inside if r[2] == r[2]), default=None)}
        if self.unparsed:
            out["unparsed_lines"] = self.unparsed
        return out


# --------------------------------------------------------------------------
# distributed plumbing (weak scaling: every rank runs its own replica)
# --------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float across the process group (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def headline_config(world: int) -> dict:
    """The workload description, identical in both arms."""
    return {"workload": WORKLOAD, "B": B, "H": H, "Nq": N, "Nk": N, "d": D, "causal": True,
            "per_gpu_batch": "one (B=1, H=32) batch per rank",
            "l2": "inputs larger than L2 (Q+K+V+O = 256 MiB > 129 MB); no flush in the timed loop",
            "parallelism": f"replicas x{world} (independent batches, no collective)"}


def repeats_for(floor_s: float, steps: int, step_ms: float) -> int:
    """How many times the K-step loop runs so that the timed region lasts at least floor_s."""
    if floor_s <= 0 or step_ms <= 0:
        return 1
    return max(1, math.ceil(floor_s * 1e3 / (steps * step_ms)))


# --------------------------------------------------------------------------
# GPU timing helpers
# --------------------------------------------------------------------------
def time_launches(fn, steps, warmup, flush=None, min_seconds=0.0, max_launches=4000):
    """Run fn() warmup times, then at least `steps` times and for at least min_seconds, with CUDA
    events around each launch on the current stream; returns per-launch milliseconds.  flush()
    (outside the events) evicts L2."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    t0 = time.perf_counter()
    while len(times) < steps or (time.perf_counter() - t0 < min_seconds and len(times) < max_launches):
        if flush is not None:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    return times


# --------------------------------------------------------------------------
# workloads: each builds its inputs on `dev` and returns a Case; the same table serves the
# components of the bench line and `--case NAME` (one workload under a profiler)
# --------------------------------------------------------------------------
class Case:
    def __init__(self, fn, work, unit, bound, workload, flush=True, launches=1, **extra):
        self.fn, self.work, self.unit, self.bound, self.workload = fn, work, unit, bound, workload
        self.flush, self.launches, self.extra = flush, launches, extra


def _case_attn_causal(oa, si, torch, dev, batch):
    q, k, v = si.attn_inputs(B, H, N, N, D, torch.bfloat16, seed=0, device=dev)
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)
    return Case(lambda: oa.attn_fwd(q, k, v, causal=True, out=o, lse=lse), causal_attn_flops(B, H, N, D), "TFLOP/s",
                "tensor", WORKLOAD)


def _case_softmax(oa, si, torch, dev, batch):
    x, *_ = si.softmax_input(4096, 32768, seed=0)
    x = x.to(dev)
    y, lse = torch.empty_like(x), torch.empty(4096, dtype=torch.float32, device=dev)
    return Case(lambda: oa.softmax_rows(x, y=y, lse=lse), softmax_bytes(4096, 32768), "GB/s", "hbm",
                "row softmax + LSE fp32 [4096, 32768], N(0,1)*4, 1% rows -inf, 10% -inf prefix")


def _case_softmax_wide(oa, si, torch, dev, batch):
    rows, cols = 256, 262144
    x, *_ = si.softmax_input(rows, cols, seed=0)
    x = x.to(dev)
    y, lse = torch.empty_like(x), torch.empty(rows, dtype=torch.float32, device=dev)
    return Case(lambda: oa.softmax_rows(x, y=y, lse=lse), softmax_bytes(rows, cols), "GB/s", "hbm",
                f"row softmax + LSE fp32 [{rows}, {cols}] (rows wider than a cluster's registers: 16 CTAs of a "
                "cluster per row, each reading its 64 KB slice twice, the second time from L2), N(0,1)*4, 1% rows "
                "-inf, 10% -inf prefix")


def _case_attn_noncausal(oa, si, torch, dev, batch):
    q, k, v = si.attn_inputs(4, 16, 4096, 4096, 64, torch.bfloat16, seed=0, device=dev)
    o, lse = torch.empty_like(q), torch.empty((4, 16, 4096), dtype=torch.float32, device=dev)
    return Case(lambda: oa.attn_fwd(q, k, v, out=o, lse=lse), dense_attn_flops(4, 16, 4096, 4096, 64), "TFLOP/s",
                "tensor", "non-causal attention fwd bf16 B=4 H=16 N=4096 d=64")


def _case_decode(oa, si, torch, dev, batch):
    b = batch or 32
    q, k, v = si.attn_inputs(b, 32, 1, 32768, 128, torch.bfloat16, seed=0, device=dev)
    kv_len = si.decode_kv_len(b, 32768, seed=0)
    kvd = kv_len.to(dev)
    o, lse = torch.empty_like(q), torch.empty((b, 32, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(oa.splitkv_workspace_bytes(b, 32, 1, 128, 64), dtype=torch.uint8, device=dev)
    return Case(lambda: oa.attn_splitkv(q, k, v, 64, kv_len=kvd, out=o, lse=lse, workspace=ws),
                decode_bytes(b, 32, 128, int(kv_len.sum())), "GB/s", "hbm",
                f"split-KV decode bf16 B={b} H=32 Nq=1 Nk=32768 d=128, 64 chunks of 512, 5% of sequences "
                f"truncated (inputs {b * 32 * 32768 * 128 * 4 / 1e9:.1f} GB)", flush=False, launches=2)


def _case_decode_gqa(oa, si, torch, dev, batch):
    b = batch or 32
    q, k, v = si.attn_inputs_gqa(b, 32, 8, 1, 32768, 128, torch.bfloat16, seed=0, device=dev)
    kv_len = si.decode_kv_len(b, 32768, seed=0)
    kvd = kv_len.to(dev)
    o, lse = torch.empty_like(q), torch.empty((b, 32, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(oa.splitkv_workspace_bytes(b, 32, 1, 128, 64), dtype=torch.uint8, device=dev)
    return Case(lambda: oa.attn_splitkv(q, k, v, 64, kv_len=kvd, out=o, lse=lse, workspace=ws),
                decode_bytes(b, 32, 128, int(kv_len.sum()), h_kv=8), "GB/s", "hbm",
                f"decode bf16 over a grouped KV cache B={b} H=32 H_kv=8 Nq=1 Nk=32768 d=128, 5% of sequences "
                "truncated, through oa_attn_splitkv_gqa: each group's 4 queries run as the rows of the "
                "tensor-core forward (no key split; num_splits and the workspace are unused)")


def _case_decode_gqa_4tok(oa, si, torch, dev, batch):
    b, nq = batch or 32, 4
    q, k, v = si.attn_inputs_gqa(b, 32, 8, nq, 32768, 128, torch.bfloat16, seed=0, device=dev)
    kv_len = si.decode_kv_len(b, 32768, seed=0)
    kvd = kv_len.to(dev)
    o, lse = torch.empty_like(q), torch.empty((b, 32, nq), dtype=torch.float32, device=dev)
    return Case(lambda: oa.attn_fwd(q, k, v, causal=True, kv_len=kvd, out=o, lse=lse),
                decode_bytes(b, 32, 128, int(kv_len.sum()), h_kv=8, nq=nq), "GB/s", "hbm",
                f"multi-token decode bf16: {nq} new tokens per sequence (causal, at the end of the cache) against a "
                f"grouped KV cache B={b} H=32 H_kv=8 Nk=32768 d=128, 5% of sequences truncated; each group's 4 heads "
                f"x {nq} tokens run as 16 rows of one plane of the tensor-core forward")


def _case_attn_varlen(oa, si, torch, dev, batch):
    lens = si.varlen_lengths(16, 8192, seed=0, min_len=1024)
    q, k, v, cq, ck = si.varlen_inputs(lens, lens, 32, 8, 128, torch.bfloat16, seed=0, device=dev)
    cq, ck = cq.to(dev), ck.to(dev)
    o, lse = torch.empty_like(q), torch.empty((q.shape[0], 32), dtype=torch.float32, device=dev)
    mx = max(lens)
    return Case(lambda: oa.attn_fwd_varlen(q, k, v, cq, ck, mx, mx, causal=True, out=o, lse=lse),
                varlen_causal_flops(lens, 32, 128), "TFLOP/s", "tensor",
                f"causal attention fwd bf16 over 16 packed sequences, lengths U[1024, 8192] (total {sum(lens)} "
                "tokens), H=32 H_kv=8 d=128")


def _case_prefill_kv_cache(oa, si, torch, dev, batch):
    b, h, hkv, nq, nk, d = batch or 8, 32, 8, 2048, 32768, 128
    q, k, v = si.attn_inputs_gqa(b, h, hkv, nq, nk, d, torch.bfloat16, seed=0, device=dev)
    o, lse = torch.empty_like(q), torch.empty((b, h, nq), dtype=torch.float32, device=dev)
    return Case(lambda: oa.attn_fwd(q, k, v, causal=True, out=o, lse=lse), kvcache_causal_flops(b, h, nq, nk, d),
                "TFLOP/s", "tensor",
                f"chunked prefill: causal attention fwd bf16 of {nq} new queries against a {nk}-key cache (the "
                f"queries are the last positions), B={b} H={h} H_kv={hkv} d={d}; FLOPs over visible pairs only "
                f"(K/V {b * hkv * nk * d * 4 / 2**30:.1f} GiB > L2)", flush=False)


def _bwd_case(oa, si, torch, dev, b, h, hkv, n, d, causal, workload):
    q, k, v = si.attn_inputs_gqa(b, h, hkv, n, n, d, torch.bfloat16, seed=0, device=dev)
    do = si.randn((b, h, n, d), 3, torch.bfloat16, dev)
    o, lse = oa.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(oa.attn_bwd_workspace_bytes(b, h, n, d), dtype=torch.uint8, device=dev)
    fl = causal_attn_bwd_flops(b, h, n, d) if causal else dense_attn_bwd_flops(b, h, n, n, d)
    return Case(lambda: oa.attn_bwd(q, k, v, o, lse, do, causal=causal, dq=dq, dk=dk, dv=dv, workspace=ws), fl,
                "TFLOP/s", "tensor", workload, launches=3)


def _case_bwd_causal(oa, si, torch, dev, batch):
    return _bwd_case(oa, si, torch, dev, 1, 32, 32, 8192, 128, True,
                     "causal attention bwd bf16 B=1 H=32 N=8192 d=128 (dQ, dK, dV from Q, K, V, O, LSE, dO)")


def _case_bwd_causal_gqa(oa, si, torch, dev, batch):
    return _bwd_case(oa, si, torch, dev, 1, 32, 8, 8192, 128, True,
                     "causal attention bwd bf16 B=1 H=32 H_kv=8 N=8192 d=128")


def _case_bwd_noncausal_d64(oa, si, torch, dev, batch):
    return _bwd_case(oa, si, torch, dev, 4, 16, 16, 4096, 64, False,
                     "non-causal attention bwd bf16 B=4 H=16 N=4096 d=64 (dQ, dK, dV from Q, K, V, O, LSE, dO)")


CASES = {
    "attn_causal": _case_attn_causal,
    "softmax_rows": _case_softmax,
    "softmax_rows_wide": _case_softmax_wide,
    "attn_noncausal_d64": _case_attn_noncausal,
    "attn_splitkv_decode": _case_decode,
    "attn_decode_gqa": _case_decode_gqa,
    "attn_decode_gqa_4tok": _case_decode_gqa_4tok,
    "attn_varlen_causal_gqa": _case_attn_varlen,
    "attn_prefill_kv_cache": _case_prefill_kv_cache,
    "attn_bwd_causal": _case_bwd_causal,
    "attn_bwd_causal_gqa": _case_bwd_causal_gqa,
    "attn_bwd_noncausal_d64": _case_bwd_noncausal_d64,
}
COMPONENTS = [n for n in CASES if n != "attn_causal"]


def components(oa, dev, peaks, peak_kind, steps, min_seconds):
    """Each hot-path kernel other than the headline one, timed alone (L2 flushed between launches
    unless its inputs are far larger than L2) for at least min_seconds."""
    import torch

    import synth_inputs as si

    out = {}
    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)

    for name in COMPONENTS:
        c = CASES[name](oa, si, torch, dev, None)
        t = time_launches(c.fn, steps, 3, flush if c.flush else None, min_seconds)
        ms = statistics.mean(t)
        if c.unit == "GB/s":
            val, peak = c.work / (ms * 1e-3) / 1e9, peaks["hbm_gbs"]
            work = {"algorithmic_bytes": c.work}
        else:
            val, peak = c.work / (ms * 1e-3) / 1e12, peaks["bf16_tflops"]
            work = {"algorithmic_flops": c.work}
        out[name] = {"workload": c.workload, "ms": ms, "launches_timed": len(t), "value": val, "unit": c.unit,
                     "bound": c.bound, "peak": peak, "frac": val / peak, "peak_kind": peak_kind,
                     "launches_per_call": c.launches, "l2_flushed": c.flush, **work, **c.extra}
        del c
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    oa.sync_status()
    del flush_buf
    torch.cuda.empty_cache()
    return out


def run_case(name, reps, batch):
    """One workload on cuda:0: one launch, then `reps` timed launches (for a profiler's launch list)."""
    import torch

    import online_softmax_attention_tiled_gb300 as oa
    import synth_inputs as si

    if name not in CASES:
        raise SystemExit(f"unknown case {name}; cases: {', '.join(CASES)}")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    c = CASES[name](oa, si, torch, dev, batch)
    t = time_launches(c.fn, reps, 1)
    oa.sync_status()
    ms = statistics.mean(t)
    val = c.work / (ms * 1e-3) / (1e9 if c.unit == "GB/s" else 1e12)
    print(f"{name}: {ms:.4f} ms per call over {reps} calls, {val:.1f} {c.unit} ({c.workload})")


# --------------------------------------------------------------------------
# CPU oracle baseline (bounded sample of the headline workload)
# --------------------------------------------------------------------------
def oracle_sample(budget_s=12.0, seed=0):
    """Times the fp64 oracle on randomly sampled rows of the causal workload, growing the
    sample until it runs for a few seconds.  Returns (TFLOP/s, threads, description)."""
    import numpy as np
    import torch

    import oracle
    import synth_inputs as si

    q, k, v = si.attn_inputs(B, H, N, N, D, torch.bfloat16, seed=seed)
    bits = [t.contiguous().view(torch.int16).numpy().view(np.uint16) for t in (q, k, v)]
    threads = os.cpu_count() or 1
    g = torch.Generator().manual_seed(seed + 99)
    nrows = 256
    spent = 0.0
    while True:
        rows = torch.randint(0, B * H * N, (nrows,), generator=g).numpy()
        i = rows % N
        flops = float(np.sum(4.0 * D * (i + 1)))
        t0 = time.perf_counter()
        oracle.attention(*bits, causal=True, rows=rows, nthreads=threads)
        dt = time.perf_counter() - t0
        spent += dt
        if dt >= budget_s / 3 or spent >= budget_s or nrows >= 1 << 22:
            break
        nrows *= 4
    desc = (f"{nrows} random query rows of the causal B1 H32 N8192 d128 workload, "
            f"{flops / 1e9:.2f} GFLOP, {dt:.2f} s, {threads} threads")
    return flops / dt / 1e12, threads, desc


# --------------------------------------------------------------------------
# main
# --------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--components", dest="components", action="store_true", default=True)
    ap.add_argument("--no-components", dest="components", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false", default=True)
    ap.add_argument("--min-seconds", type=float, default=3.0,
                    help="time floor of the headline's timed region (the K-step loop repeats until reached)")
    ap.add_argument("--component-seconds", type=float, default=0.6, help="time floor of each component")
    ap.add_argument("--case", default=None, help="run one workload only (see CASES), for a profiler")
    ap.add_argument("--reps", type=int, default=2, help="--case: timed calls after one warm-up call")
    ap.add_argument("--batch", type=int, default=None, help="--case: batch of the decode workloads (default 32)")
    args = ap.parse_args()
    if args.case is not None:
        return run_case(args.case, args.reps, args.batch)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if world != args.gpus:
        if world > 1 or args.gpus > 1:
            ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}; launch N>1 with torchrun")

    if args.impl == "reference":
        return main_reference(args, world, rank)

    import torch

    import online_softmax_attention_tiled_gb300 as oa
    import synth_inputs as si

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    oa.load()
    peaks, peak_kind = load_peaks()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count

    q, k, v = si.attn_inputs(B, H, N, N, D, torch.bfloat16, seed=rank)
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        oa.attn_fwd(q, k, v, causal=True, out=o, lse=lse)

    with ClockSampler(local) as clocks:
        # warm-up, timed once to size the repeats of the K-step loop
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        step()
        w0.record(stream)
        for _ in range(args.warmup - 1):
            step()
        w1.record(stream)
        torch.cuda.synchronize()
        oa.sync_status()
        warm_ms = w0.elapsed_time(w1) / max(1, args.warmup - 1)
        repeats = int(max_over_ranks(float(repeats_for(args.min_seconds, args.steps, warm_ms)), world, dev))
        clocks.wait_first()

        # ---- timed region: the K-step loop, `repeats` times; one event pair per launch ----
        n_timed = repeats * args.steps
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_timed)]
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        t_wall0 = time.time()
        start.record(stream)
        for a, b in ev:
            a.record(stream)
            step()
            b.record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.time()
        barrier(world)
    oa.sync_status()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), world, dev)
    per_launch = [a.elapsed_time(b) for a, b in ev]
    launch_ms = statistics.mean(per_launch)
    flops = causal_attn_flops(B, H, N, D)
    value = world * n_timed * flops / (elapsed_ms * 1e-3) / 1e12
    achieved = flops / (launch_ms * 1e-3) / 1e12
    clock_summary = clocks.summary(t_wall0, t_wall1)
    sm_mhz = clock_summary.get("sm_mhz")
    clock_norm = None
    if sm_mhz:
        hw_peak = sm_count * BF16_FLOP_PER_SM_CLOCK * sm_mhz * 1e6 / 1e12
        clock_norm = {"sm_mhz_median": sm_mhz, "sm_count": sm_count,
                      "tflops_per_sm_ghz": achieved / (sm_mhz / 1e3),
                      "hw_peak_at_clock_tflops": hw_peak, "frac_of_hw_peak_at_clock": achieved / hw_peak,
                      "basis": f"{BF16_FLOP_PER_SM_CLOCK} dense bf16 FLOP per SM per clock (one 128x128x16 MMA "
                               "per 64 cycles) x SMs x median SM clock during the timed region"}

    # ---- end to end through the C ABI on host buffers: pinned Q/K/V in, pinned O/LSE out; the
    # library copies in, computes and copies out in pieces that overlap ----
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    e2e_ws = torch.empty(oa.attn_fwd_host_workspace_bytes(torch.bfloat16, B, H, H, N, N, D), dtype=torch.uint8,
                         device=dev)
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        oa.attn_fwd_host(qh, kh, vh, causal=True, out=oh, lse=lh, workspace=e2e_ws)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b), world, dev) / e2e_steps
    oa.sync_status()
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size()
    # the host result must be the device result
    oa.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    e2e_ok = bool(torch.equal(oh, o.cpu()) and torch.equal(lh, lse.cpu()))
    del qh, kh, vh, oh, lh, e2e_ws

    comps = None
    if args.components and rank == 0:
        del q, k, v, o, lse
        torch.cuda.empty_cache()
        comps = components(oa, dev, peaks, peak_kind, max(5, min(args.steps, 20)), args.component_seconds)

    cpu = None
    if args.cpu_baseline and rank == 0 and world == 1:
        tf, threads, desc = oracle_sample()
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc}

    barrier(world)
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": elapsed_ms / n_timed,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic: seeded N(0,1) Q/K/V cast to bf16 (no dataset is named)",
            "config": headline_config(world),
            "timing": {"repeats_of_k_steps": repeats, "timed_steps": n_timed, "timed_region_s": elapsed_ms / 1e3,
                       "min_seconds": args.min_seconds,
                       "rule": "the K-step loop repeats until the timed region reaches min_seconds; "
                               "per-step figures come from all timed steps"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"], "traffic": profiled_traffic(),
                         "peak_kind": f"{peak_kind} bf16 dense burst", "launch_ms": launch_ms,
                         "algorithmic_flops_per_launch": flops, "clock_normalised": clock_norm},
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "path": "oa_attn_fwd_host: pinned host Q/K/V in, O/LSE out; copies and kernels of 4 tapered "
                            "pieces overlapped", "matches_device_result": e2e_ok},
            "gpu_launches": n_timed,
            "clocks": clock_summary,
            "cpu_baseline": cpu,
            "components": comps,
            "kernel_source_digest": kernel_source_digest(),
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle, each step a bounded sample of the workload."""
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    import synth_inputs as si

    q, k, v = si.attn_inputs(B, H, N, N, D, torch.bfloat16, seed=0)
    bits = [t.contiguous().view(torch.int16).numpy().view(np.uint16) for t in (q, k, v)]
    threads = os.cpu_count() or 1
    g = torch.Generator().manual_seed(7)
    rows_per_step = 512

    def step():
        rows = torch.randint(0, B * H * N, (rows_per_step,), generator=g).numpy()
        oracle.attention(*bits, causal=True, rows=rows, nthreads=threads)
        return float(np.sum(4.0 * D * (rows % N + 1)))

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    flops = sum(step() for _ in range(args.steps))
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    desc = f"each step: {rows_per_step} random query rows of the causal workload ({threads} threads, fp64)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


if __name__ == "__main__":
    main()
