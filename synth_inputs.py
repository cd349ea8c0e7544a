"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers and places -inf masks; it holds none of
the softmax or attention arithmetic, so both the CPU oracle and the CUDA path
can be fed from it without sharing any of the method's code.

Recipe (all seeded; tensor k of a call uses seed + k):
  * attention Q, K, V: N(0, 1) drawn in fp32, then rounded to nearest-even into
    the requested dtype (bf16 or fp32); K and V may have fewer heads than Q
    (grouped heads), or be packed token-major [tokens, heads, d] with int32
    offsets of a list of sequence lengths (variable-length batches);
  * row-softmax X: N(0, 1) * 4 in fp32; round(1% of rows) fully -inf; another
    10% of rows (disjoint, chosen by a seeded permutation) get a -inf prefix of
    length uniform in [1, cols - 1];
  * decode key lengths: ceil(5% of the batch) sequences, chosen by a seeded
    permutation, get a length uniform in [1, Nk]; the rest keep Nk;
  * the [8, 37] lesson matrix: N(0, 1) * 10 with row 1 [:20] = -inf and row 2
    entirely -inf, split into column chunks [5, 1, 13, 8, 10].
"""
from __future__ import annotations

import itertools
import math

import torch

LESSON_CHUNKS = (5, 1, 13, 8, 10)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, seed: int, dtype=torch.float32, device="cpu", mul: float = 1.0) -> torch.Tensor:
    """N(0,1)*mul drawn in fp32 with a fresh seeded generator, then cast (RNE) to dtype."""
    t = torch.randn(*shape, generator=_gen(seed, device), dtype=torch.float32, device=device)
    if mul != 1.0:
        t.mul_(mul)
    return t.to(dtype)


def attn_inputs(B, H, Nq, Nk, d, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Q [B,H,Nq,d], K and V [B,H,Nk,d] ~ N(0,1), seeds seed, seed+1, seed+2."""
    q = randn((B, H, Nq, d), seed, dtype, device)
    k = randn((B, H, Nk, d), seed + 1, dtype, device)
    v = randn((B, H, Nk, d), seed + 2, dtype, device)
    return q, k, v


def attn_inputs_gqa(B, H, Hkv, Nq, Nk, d, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Q [B,H,Nq,d], K and V [B,Hkv,Nk,d] ~ N(0,1) (grouped key/value heads)."""
    q = randn((B, H, Nq, d), seed, dtype, device)
    k = randn((B, Hkv, Nk, d), seed + 1, dtype, device)
    v = randn((B, Hkv, Nk, d), seed + 2, dtype, device)
    return q, k, v


def varlen_lengths(n, max_len, seed=0, min_len=0):
    """n sequence lengths, uniform on [min_len, max_len], as a Python list."""
    g = _gen(seed)
    return torch.randint(min_len, max_len + 1, (n,), generator=g, dtype=torch.int64).tolist()


def varlen_inputs(lq, lk, H, Hkv, d, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Packed token-major Q [sum lq, H, d], K and V [sum lk, Hkv, d] ~ N(0,1), and the int32 offsets
    cu_q = [0, lq0, lq0 + lq1, ...], cu_k likewise."""
    cu_q = torch.tensor([0] + list(itertools.accumulate(lq)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(itertools.accumulate(lk)), dtype=torch.int32)
    q = randn((int(cu_q[-1]), H, d), seed, dtype, device)
    k = randn((int(cu_k[-1]), Hkv, d), seed + 1, dtype, device)
    v = randn((int(cu_k[-1]), Hkv, d), seed + 2, dtype, device)
    return q, k, v, cu_q, cu_k


def softmax_input(rows, cols, seed=0, mul=4.0, frac_full=0.01, frac_prefix=0.10, device="cpu"):
    """X fp32 [rows, cols] ~ N(0,1)*mul with fully -inf rows and -inf prefixes.

    Returns (X, full_rows, prefix_rows, prefix_lens) -- the latter three as CPU tensors.
    """
    x = randn((rows, cols), seed, torch.float32, device, mul)
    g = _gen(seed + 1)
    perm = torch.randperm(rows, generator=g)
    n_full = int(round(frac_full * rows))
    n_pre = int(round(frac_prefix * rows))
    full_rows = perm[:n_full].sort().values
    prefix_rows = perm[n_full:n_full + n_pre].sort().values
    if cols > 1:
        prefix_lens = torch.randint(1, cols, (prefix_rows.numel(),), generator=g)
    else:
        prefix_lens = torch.zeros(prefix_rows.numel(), dtype=torch.int64)
    neg = float("-inf")
    if n_full:
        x[full_rows.to(x.device)] = neg
    for r, n in zip(prefix_rows.tolist(), prefix_lens.tolist()):
        if n > 0:
            x[r, :n] = neg
    return x, full_rows, prefix_rows, prefix_lens


def decode_kv_len(B, Nk, seed=0, frac=0.05) -> torch.Tensor:
    """int32 [B]: Nk for most sequences, ceil(frac*B) of them truncated to U[1, Nk]."""
    g = _gen(seed)
    kv = torch.full((B,), Nk, dtype=torch.int32)
    n_trunc = int(math.ceil(frac * B))
    idx = torch.randperm(B, generator=g)[:n_trunc]
    lens = torch.randint(1, Nk + 1, (n_trunc,), generator=g, dtype=torch.int64)
    kv[idx] = lens.to(torch.int32)
    return kv


def lesson_matrix(seed=0) -> torch.Tensor:
    """[8, 37] fp32 N(0,1)*10, row 1 [:20] = -inf, row 2 all -inf."""
    x = randn((8, 37), seed, torch.float32, "cpu", 10.0)
    x[1, :20] = float("-inf")
    x[2, :] = float("-inf")
    return x


def sample_rows(n_rows: int, count: int, seed=0, tile: int = 128, must=()) -> torch.Tensor:
    """Sorted unique row indices in [0, n_rows): the first/last rows, each tile
    boundary pair (t*tile - 1, t*tile), any rows in `must`, and seeded random fill
    up to `count` rows."""
    picks = {0, min(1, n_rows - 1), n_rows - 1}
    for t in range(1, (n_rows + tile - 1) // tile):
        b = t * tile
        if b < n_rows:
            picks.update((b - 1, b))
    picks.update(int(m) for m in must if 0 <= int(m) < n_rows)
    if len(picks) < count:
        g = _gen(seed)
        extra = torch.randperm(n_rows, generator=g)[:count].tolist()
        for e in extra:
            if len(picks) >= count:
                break
            picks.add(e)
    return torch.tensor(sorted(picks), dtype=torch.int64)
