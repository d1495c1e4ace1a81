"""Build libagmm.so (the C-ABI library) in-tree with nvcc for sm_103a.

Cross-compiles without a GPU.  One translation unit, one -gencode, static
cudart; the result lands next to this file and is git-ignored.  The
bounds-checked variant libagmm_debug.so (-DAGMM_DEBUG: every flag, per-tile
word, shard-row and staging index is checked against its buffer; a violation
is recorded as AG_ERR_BOUNDS and the access skipped) is compiled alongside it,
in parallel, from the same sources.
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
DEBUG_LIB_PATH = os.path.join(PKG, "libagmm_debug.so")
VARIANTS = {"release": (LIB_PATH, ()), "debug": (DEBUG_LIB_PATH, ("-DAGMM_DEBUG",))}
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


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(s) > t for s in SOURCES)


def build(force: bool = False, verbose: bool = False, extra=(),
          variants=("release", "debug")) -> str:
    """Compile the variants that are missing or older than their sources (all
    of them with `force` or `extra` flags), in parallel.  Returns the release
    library's path."""
    jobs = []
    for v in variants:
        path, flags = VARIANTS[v]
        if not force and not extra and not is_stale(path):
            continue
        tmp = path + f".tmp{os.getpid()}"
        cmd = nvcc_command(tmp, (*flags, *extra))
        proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
        jobs.append((v, path, tmp, cmd, proc))
    failed = []
    for v, path, tmp, cmd, proc in jobs:
        out, err = proc.communicate()
        if verbose or proc.returncode != 0:
            print(" ".join(cmd))
            print(out, err)
        if proc.returncode != 0:
            failed.append((v, proc.returncode))
            continue
        os.replace(tmp, path)
    if failed:
        raise RuntimeError(f"nvcc failed: {failed}")
    return LIB_PATH


if __name__ == "__main__":
    import sys
    build(force=True, verbose=True, extra=sys.argv[1:])
