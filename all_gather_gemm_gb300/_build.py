"""Build libagmm.so (the C-ABI library) in-tree with nvcc for sm_103a.

Cross-compiles without a GPU.  One translation unit, one -gencode, static
cudart; the result lands next to this file and is git-ignored.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libagmm.so")
SOURCES = [os.path.join(CSRC, f) for f in ("agmm.cu", "kernels.cuh", "ptx.cuh")] + [
    os.path.join(INCLUDE, "agmm.h")]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libagmm")


def nvcc_command(out: str, extra=()) -> list:
    return [nvcc_path(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-shared", "-I", INCLUDE, *extra, "-o", out, os.path.join(CSRC, "agmm.cu")]


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(s) > t for s in SOURCES)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile if missing or older than its sources.  Returns the library path."""
    if not force and not extra and not is_stale():
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp, extra)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        print(" ".join(cmd))
        print(res.stdout, res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed with exit code {res.returncode}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    build(force=True, verbose=True, extra=sys.argv[1:])
