"""CPU oracle for the all-gather matmul -- TEST INFRASTRUCTURE, not product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never calls it, and it shares
no code with the CUDA path: the arithmetic lives in ``agmm_oracle.c`` (plain
C, built with gcc), and this module only marshals numpy arrays to it.

What it computes ("Add all gather matmul benchmark", pytorch/helion PR #400,
statement of the op; "Fused all-gather+GEMM HBM-buffer kernel for iris.ops",
ROCm/iris #346, section "New kernel", for the optional bias):

    a_gathered = concat_rows(a_shards[0], ..., a_shards[D-1])
    out_f32[i, j] = sum_{k=0..K-1} f32(a[i, k]) * f32(b[k, j])   (fp32, k increasing)
                    (+ bias[j], fp32)
    out = round_to_nearest_even_16bit(out_f32)

16-bit arrays are passed as ``numpy.uint16`` bit patterns; ``dtype`` is
``"bf16"`` or ``"fp16"``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "agmm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libagmm_oracle.so")
_DTYPES = {"bf16": 0, "fp16": 1}
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU needed).  Returns the .so path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f32p = ctypes.POINTER(ctypes.c_float)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_fp16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f32_to_fp16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_fp16.restype = ctypes.c_uint16
        lib.oracle_to_f32.argtypes = [u16p, ctypes.c_int64, ctypes.c_int, f32p]
        lib.oracle_to_f32.restype = None
        lib.oracle_from_f32.argtypes = [f32p, ctypes.c_int64, ctypes.c_int, u16p]
        lib.oracle_from_f32.restype = None
        lib.oracle_all_gather.argtypes = [ctypes.POINTER(u16p), ctypes.c_int,
                                          ctypes.c_int64, ctypes.c_int64, u16p]
        lib.oracle_all_gather.restype = None
        lib.oracle_gemm_rows.argtypes = [u16p, ctypes.c_int64, ctypes.c_int64, u16p,
                                         ctypes.c_int64, f32p, ctypes.c_int, i64p,
                                         ctypes.c_int64, f32p, u16p, f32p, ctypes.c_int]
        lib.oracle_gemm_rows.restype = ctypes.c_int
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f32.restype = ctypes.c_float
        lib.oracle_e4m3_to_f32_array.argtypes = [u8p, ctypes.c_int64, f32p]
        lib.oracle_e4m3_to_f32_array.restype = None
        lib.oracle_all_gather_bytes.argtypes = [ctypes.POINTER(u8p), ctypes.c_int,
                                                ctypes.c_int64, ctypes.c_int64, u8p]
        lib.oracle_all_gather_bytes.restype = None
        lib.oracle_gemm_rows_fp8.argtypes = [u8p, ctypes.c_int64, ctypes.c_int64, u8p,
                                             ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                                             f32p, i64p, ctypes.c_int64, f32p, u16p, f32p,
                                             ctypes.c_int]
        lib.oracle_gemm_rows_fp8.restype = ctypes.c_int
        _lib = lib
        return lib


def _u16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError(f"expected uint16 bit patterns, got {x.dtype}")
    return x


def _ptr(x: np.ndarray, ctype):
    return x.ctypes.data_as(ctypes.POINTER(ctype))


def to_f32(bits, dtype: str) -> np.ndarray:
    """Widen 16-bit patterns to fp32 (exact)."""
    bits = _u16(bits)
    out = np.empty(bits.shape, np.float32)
    _load().oracle_to_f32(_ptr(bits, ctypes.c_uint16), bits.size, _DTYPES[dtype],
                          _ptr(out, ctypes.c_float))
    return out


def from_f32(x, dtype: str) -> np.ndarray:
    """Round fp32 values to 16-bit patterns, round-to-nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_from_f32(_ptr(x, ctypes.c_float), x.size, _DTYPES[dtype],
                            _ptr(out, ctypes.c_uint16))
    return out


def all_gather(shards) -> np.ndarray:
    """Row concatenation of D equally sized [m_per_shard, K] shards."""
    shards = [_u16(s) for s in shards]
    D = len(shards)
    mps, K = shards[0].shape
    for s in shards:
        if s.shape != (mps, K):
            raise ValueError("all shards must have the same shape")
    out = np.empty((D * mps, K), np.uint16)
    arr = (ctypes.POINTER(ctypes.c_uint16) * D)(*[_ptr(s, ctypes.c_uint16) for s in shards])
    _load().oracle_all_gather(arr, D, mps, K, _ptr(out, ctypes.c_uint16))
    return out


def gemm_rows(a, b, bias=None, *, dtype: str, rows=None, want_abs: bool = True,
              nthreads: int = 0):
    """Rows ``rows`` of a @ b (+ bias).  Returns (out_f32, out_bits, abs_ab, threads).

    ``abs_ab[t, j] = sum_k |a[rows[t], k]| |b[k, j]|`` (the scale in the parity
    tolerance), or None when ``want_abs`` is False.
    """
    a = _u16(a)
    b = _u16(b)
    M, K = a.shape
    K2, N = b.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= M):
        raise IndexError("row index out of range")
    nr = rows.size
    out_f32 = np.empty((nr, N), np.float32)
    out = np.empty((nr, N), np.uint16)
    abs_ab = np.empty((nr, N), np.float32) if want_abs else None
    bias_p = None
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        if bias.shape != (N,):
            raise ValueError("bias must have shape [N]")
        bias_p = _ptr(bias, ctypes.c_float)
    threads = _load().oracle_gemm_rows(
        _ptr(a, ctypes.c_uint16), M, K, _ptr(b, ctypes.c_uint16), N, bias_p,
        _DTYPES[dtype], _ptr(rows, ctypes.c_int64), nr, _ptr(out_f32, ctypes.c_float),
        _ptr(out, ctypes.c_uint16),
        _ptr(abs_ab, ctypes.c_float) if abs_ab is not None else None, nthreads)
    return out_f32, out, abs_ab, threads


def ag_matmul(shards, b, bias=None, *, dtype: str, rows=None, want_abs: bool = True,
              nthreads: int = 0):
    """The whole op: gather the shards, then the GEMM on rows ``rows``.

    Returns ``(a_gathered, out_f32, out_bits, abs_ab)``.
    """
    a = all_gather(shards)
    out_f32, out, abs_ab, _ = gemm_rows(a, b, bias, dtype=dtype, rows=rows,
                                        want_abs=want_abs, nthreads=nthreads)
    return a, out_f32, out, abs_ab


def within_tolerance(got_f32, ref_f32, abs_ab, rel: float = 1e-2, atol: float = 1e-3):
    """The parity bound |got - ref| <= rel * (|a|.|b|)_ij + atol, elementwise.

    Returns (ok, worst_ratio, first_bad_index or None).
    """
    got = np.asarray(got_f32, np.float64)
    ref = np.asarray(ref_f32, np.float64)
    bound = rel * np.asarray(abs_ab, np.float64) + atol
    err = np.abs(got - ref)
    bad = ~(err <= bound)  # NaN counts as a violation
    ratio = float(np.nanmax(err / bound)) if err.size else 0.0
    if bad.any():
        return False, ratio, tuple(int(v) for v in np.argwhere(bad)[0])
    return True, ratio, None


# ---------------------------------------------------------------- FP8 E4M3
# An extension the pages do not cover: 8-bit inputs with per-tensor scales,
#     out_f32[i, j] = (scale_a * scale_b) * sum_k f32(a[i, k]) * f32(bt[j, k])
#                     (+ bias[j]),   out = bf16(out_f32)
# with b given transposed (bt = [N, K]); sums in fp32, k increasing.


def _u8(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint8:
        raise TypeError(f"expected uint8 bit patterns, got {x.dtype}")
    return x


def e4m3_to_f32(bits) -> np.ndarray:
    """Decode E4M3 bit patterns to fp32 (exact)."""
    bits = _u8(bits)
    out = np.empty(bits.shape, np.float32)
    _load().oracle_e4m3_to_f32_array(_ptr(bits, ctypes.c_uint8), bits.size,
                                     _ptr(out, ctypes.c_float))
    return out


def all_gather_bytes(shards) -> np.ndarray:
    """Row concatenation of D equally shaped 2-D byte arrays (any element type
    stored as uint8)."""
    shards = [_u8(s) for s in shards]
    D = len(shards)
    mps, row = shards[0].shape
    for s in shards:
        if s.shape != (mps, row):
            raise ValueError("all shards must have the same shape")
    out = np.empty((D * mps, row), np.uint8)
    arr = (ctypes.POINTER(ctypes.c_uint8) * D)(*[_ptr(s, ctypes.c_uint8) for s in shards])
    _load().oracle_all_gather_bytes(arr, D, mps, row, _ptr(out, ctypes.c_uint8))
    return out


def gemm_rows_fp8(a, bt, scale_a: float = 1.0, scale_b: float = 1.0, bias=None, *, rows=None,
                  want_abs: bool = True, nthreads: int = 0):
    """Rows ``rows`` of scale_a*scale_b * (a @ bt.T) (+ bias) for E4M3 ``a`` [M, K]
    and ``bt`` [N, K] (uint8 bit patterns).  Returns (out_f32, out_bf16_bits,
    abs_ab, threads) with ``abs_ab = |scale_a*scale_b| * sum_k |a| |b|``."""
    a = _u8(a)
    bt = _u8(bt)
    M, K = a.shape
    N, K2 = bt.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= M):
        raise IndexError("row index out of range")
    nr = rows.size
    out_f32 = np.empty((nr, N), np.float32)
    out = np.empty((nr, N), np.uint16)
    abs_ab = np.empty((nr, N), np.float32) if want_abs else None
    bias_p = None
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        if bias.shape != (N,):
            raise ValueError("bias must be [N]")
        bias_p = _ptr(bias, ctypes.c_float)
    th = _load().oracle_gemm_rows_fp8(
        _ptr(a, ctypes.c_uint8), M, K, _ptr(bt, ctypes.c_uint8), N, float(scale_a),
        float(scale_b), bias_p, _ptr(rows, ctypes.c_int64), nr, _ptr(out_f32, ctypes.c_float),
        _ptr(out, ctypes.c_uint16), _ptr(abs_ab, ctypes.c_float) if want_abs else None,
        nthreads)
    return out_f32, out, abs_ab, th
