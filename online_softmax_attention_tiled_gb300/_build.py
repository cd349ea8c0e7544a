"""Builds liboa.so (the CUDA library behind include/oa.h) in-tree for sm_103a.

Each .cu file is compiled to an object in parallel, then linked into one
shared object next to this file.  No cmake; nvcc only.  ``build(debug=True)``
builds liboa_debug.so instead: the same sources with -DOA_DEBUG, whose kernels
check the bounds and alignment of their computed global accesses and record a
failed check in the status word (see oa_common.cuh).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "liboa.so")
DEBUG_LIB_PATH = os.path.join(PKG, "liboa_debug.so")

SOURCES = ["oa_api.cu", "tma_map.cu", "softmax_rows.cu", "lse_merge.cu", "attn_f32.cu", "attn_splitkv.cu", "attn_tc.cu",
           "attn_bwd.cu", "attn_splitkv_static.cu"]
HEADERS = ["oa_common.cuh", "oa_internal.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I" + CSRC, "-I" + INCLUDE]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA library cannot be built")
    return cand


def _inputs_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "oa.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, verbose_ptxas: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD_DIR, ("debug_" if debug else "") + os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + (["-DOA_DEBUG"] if debug else []) + \
        (["-Xptxas", "-v"] if verbose_ptxas else []) + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Compile and link liboa.so (debug: liboa_debug.so) if any input is newer than it.  Returns its
    path."""
    path = DEBUG_LIB_PATH if debug else LIB_PATH
    if not force and os.path.exists(path) and os.path.getmtime(path) >= _inputs_mtime():
        return path
    os.makedirs(BUILD_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, debug), SOURCES))
    tmp = path + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
