"""Build the CUDA library in-tree: tensor_gemm_reduce_gb300/lib/libgemm_rs.so.

One nvcc invocation for sm_103a (tcgen05 / TMA need the arch-specific target).
The library links the CUDA runtime statically and resolves the one driver call
it needs (cuTensorMapEncodeTiled) at run time, so it has no link-time
dependency on libcuda.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libgemm_rs.so")
SOURCES = [os.path.join(CSRC, "gemm_rs.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("kernels.cuh", "ptx.cuh", "schedule.h")] + [
    os.path.join(ROOT, "include", "gemm_rs.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in DEPS)


def build_library(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile the library if it is missing or older than its sources; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc_path()] + NVCC_FLAGS + list(extra_flags or []) + ["-o", tmp] + SOURCES
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed ({r.returncode}):\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))
