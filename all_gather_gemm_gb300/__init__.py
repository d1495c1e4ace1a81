"""GB300-native fused all-gather matmul: Python binding of libagmm.

Thin ctypes marshalling over the C ABI in ``include/agmm.h``; every step of
the operation runs in the library's CUDA kernels.  PyTorch only provides the
device memory and the current stream.  There is no fallback: if the compiled
library is missing, every call raises.

    a_gathered, out = ag_matmul(shards, b, bias=None, layout="k_contiguous", rank=0)

``shards`` is a list of D CUDA tensors [m_per_shard, K] (bf16 or fp16, the
D row shards of A, each its own allocation); ``b`` is [K, N] of the same
dtype; ``bias`` an optional fp32 [N].  ``a_gathered`` = concat(shards) and
``out`` = a_gathered @ b (+ bias), computed with fp32 accumulation.

FP8 (``torch.float8_e4m3fn`` shards): ``b`` is given transposed, [N, K] e4m3,
``out`` is bf16 and ``out = scale_a * scale_b * (a_gathered @ b.T) + bias``
(k-contiguous layout only).

With the environment variable ``AGMM_VARIANT=debug`` (or ``AGMM_DEBUG=1``) set
before the first call, the bounds-checked build ``libagmm_debug.so`` is loaded
instead (every
flag, per-tile word, shard-row and staging index checked on the device; a
violation is reported by ``device_error()`` as AG_ERR_BOUNDS).
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = [
    "AgmmError", "AgOptions", "ag_matmul", "ag_then_matmul", "ag_matmul_raw",
    "device_error", "workspace_size", "release_workspace", "num_sms", "library",
    "LAYOUTS", "STATUS",
]

STATUS = {0: "AG_OK", 1: "AG_ERR_INVALID_ARG", 2: "AG_ERR_UNSUPPORTED", 3: "AG_ERR_CUDA",
          4: "AG_ERR_TIMEOUT", 5: "AG_ERR_WORKSPACE", 6: "AG_ERR_TOO_LARGE", 7: "AG_ERR_BUSY",
          8: "AG_ERR_BOUNDS"}
LAYOUTS = {"k_contiguous": 0, "m_contiguous": 1}
DTYPES = {"bf16": 0, "fp16": 1, "fp8_e4m3": 2}
EXPORTS = ("ag_options_default", "ag_matmul", "ag_then_matmul", "ag_matmul_ex",
           "ag_then_matmul_ex", "ag_workspace_size", "ag_get_device_error",
           "ag_release_workspace", "ag_status_string", "ag_num_sms", "ag_matmul_noalloc",
           "ag_chunked_matmul_ex")


class AgmmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({_status_text(status)})")


class AgOptions(ctypes.Structure):
    """Mirror of ``struct ag_options``."""
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("rank", ctypes.c_int32),
        ("k_per_flag", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("inject_skip_flag", ctypes.c_int32),
        ("timeout_ns", ctypes.c_int64),
        ("trace", ctypes.c_void_p),
        ("trace_words", ctypes.c_int64),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_int64),
        ("scale_a", ctypes.c_float),
        ("scale_b", ctypes.c_float),
        ("inject_delay_ns", ctypes.c_int64),
        ("block_m", ctypes.c_int32),
        ("block_n", ctypes.c_int32),
        ("block_k", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("producer_warps", ctypes.c_int32),
    ]


_lib = None


def variant() -> str:
    """The library variant this process loads: "release", or "debug" (the
    bounds-checked build) when AGMM_VARIANT=debug or AGMM_DEBUG=1."""
    v = os.environ.get("AGMM_VARIANT", "") or ""
    if not v:
        v = "debug" if os.environ.get("AGMM_DEBUG", "0") not in ("", "0") else "release"
    if v not in _build.VARIANTS:
        raise ValueError(f"AGMM_VARIANT must be one of {sorted(_build.VARIANTS)}, not {v!r}")
    return v


def library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libagmm.so, or libagmm_debug.so under AGMM_VARIANT=debug (building
    it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    v = variant()
    path = _build.VARIANTS[v][0]
    if build_if_missing and _build.is_stale(path):
        _build.build(variants=(v,))
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} not found at {path}; build it with "
                           "__graft_entry__.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    core = [ctypes.POINTER(vp), i32, i32, i32, vp, i32, vp, vp, vp, vp]
    for name in ("ag_matmul", "ag_then_matmul"):
        getattr(lib, name).argtypes = core
        getattr(lib, name).restype = i32
    for name in ("ag_matmul_ex", "ag_then_matmul_ex"):
        getattr(lib, name).argtypes = core + [ctypes.POINTER(AgOptions)]
        getattr(lib, name).restype = i32
    lib.ag_options_default.argtypes = [ctypes.POINTER(AgOptions)]
    lib.ag_options_default.restype = None
    lib.ag_workspace_size.argtypes = [i32, i32, i32, i32, ctypes.POINTER(AgOptions)]
    lib.ag_workspace_size.restype = ctypes.c_size_t
    lib.ag_get_device_error.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.ag_get_device_error.restype = i32
    lib.ag_release_workspace.argtypes = []
    lib.ag_release_workspace.restype = i32
    lib.ag_status_string.argtypes = [i32]
    lib.ag_status_string.restype = ctypes.c_char_p
    lib.ag_num_sms.argtypes = []
    lib.ag_plan_fused.argtypes = [i32, i32, i32, i32, ctypes.POINTER(AgOptions), i32, i32,
                                  ctypes.POINTER(AgPlan)]
    lib.ag_plan_fused.restype = i32
    lib.ag_num_sms.restype = i32
    lib.ag_matmul_noalloc.argtypes = core + [ctypes.POINTER(AgOptions)]
    lib.ag_matmul_noalloc.restype = i32
    lib.ag_chunked_matmul_ex.argtypes = core + [ctypes.POINTER(AgOptions), i32]
    lib.ag_chunked_matmul_ex.restype = i32
    _lib = lib
    return lib


def _status_text(status: int) -> str:
    try:
        return library().ag_status_string(status).decode()
    except Exception:  # pragma: no cover - library unavailable while formatting
        return "?"


_DEFAULT_OPTIONS = None


def default_options() -> AgOptions:
    """A fresh ag_options filled by ag_options_default (the C side's defaults)."""
    global _DEFAULT_OPTIONS
    if _DEFAULT_OPTIONS is None:
        o = AgOptions()
        library().ag_options_default(ctypes.byref(o))
        _DEFAULT_OPTIONS = bytes(o)
    return AgOptions.from_buffer_copy(_DEFAULT_OPTIONS)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_name(t) -> str:
    import torch
    if t.dtype == torch.bfloat16:
        return "bf16"
    if t.dtype == torch.float16:
        return "fp16"
    if t.dtype == getattr(torch, "float8_e4m3fn", None):
        return "fp8_e4m3"
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16, float16 or float8_e4m3fn")


def ag_matmul_raw(fused: bool, shard_ptrs, D, m_per_shard, K, b_ptr, N, bias_ptr, ag_ptr, out_ptr,
                  stream_handle, options: AgOptions | None = None) -> int:
    """Direct call of the C entry point with integer pointers; returns the status."""
    lib = library()
    arr = (ctypes.c_void_p * max(D, 1))(*[ctypes.c_void_p(p) for p in shard_ptrs])
    args = [arr, D, m_per_shard, K, ctypes.c_void_p(b_ptr), N,
            ctypes.c_void_p(bias_ptr) if bias_ptr else None, ctypes.c_void_p(ag_ptr),
            ctypes.c_void_p(out_ptr), stream_handle]
    if options is None:
        return (lib.ag_matmul if fused else lib.ag_then_matmul)(*args)
    fn = lib.ag_matmul_ex if fused else lib.ag_then_matmul_ex
    return fn(*args, ctypes.byref(options))


TILE_OPTIONS = ("block_m", "block_n", "block_k", "stages", "producer_warps")


def _call(fused, shards, b, bias, a_gathered, out, stream, layout, rank, k_per_flag, num_sms,
          timeout_ns, inject_skip_flag, trace, workspace, chunks=0, scale_a=1.0, scale_b=1.0,
          inject_delay_ns=0, tile=None):
    import torch
    if not shards:
        raise ValueError("need at least one shard")
    D = len(shards)
    m, K = shards[0].shape
    dt = _dtype_name(b)
    fp8 = dt == "fp8_e4m3"
    if fp8:
        N, K2 = b.shape  # FP8: b is given transposed, [N, K]
    else:
        K2, N = b.shape
    for s in shards:
        if s.shape != (m, K) or s.dtype != b.dtype or not s.is_cuda or not s.is_contiguous():
            raise ValueError("shards must be contiguous CUDA tensors of one shape and b's dtype")
    if K2 != K or not b.is_cuda or not b.is_contiguous():
        raise ValueError("b must be a contiguous CUDA tensor [N, K]" if fp8
                         else "b must be a contiguous CUDA tensor [K, N]")
    M = D * m
    out_dtype = torch.bfloat16 if fp8 else b.dtype
    if a_gathered is None:
        a_gathered = torch.empty((M, K), dtype=b.dtype, device=b.device)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=b.device)
    if (a_gathered.shape != (M, K) or a_gathered.dtype != b.dtype or out.shape != (M, N)
            or out.dtype != out_dtype):
        raise ValueError("a_gathered must be [M, K] of the inputs' dtype and out [M, N] of "
                         + ("bf16" if fp8 else "the inputs' dtype"))
    if bias is not None and (bias.dtype != torch.float32 or bias.shape != (N,) or not bias.is_cuda):
        raise ValueError("bias must be a CUDA fp32 tensor [N]")
    o = default_options()
    o.dtype = DTYPES[dt]
    o.layout = LAYOUTS[layout]
    o.rank = rank
    o.k_per_flag = k_per_flag
    o.num_sms = num_sms
    o.timeout_ns = timeout_ns
    o.inject_skip_flag = inject_skip_flag
    o.scale_a = scale_a
    o.scale_b = scale_b
    o.inject_delay_ns = inject_delay_ns
    for name, value in (tile or {}).items():
        if name not in TILE_OPTIONS:
            raise TypeError(f"unknown tile option {name!r}; one of {TILE_OPTIONS}")
        setattr(o, name, value)
    if trace is not None:
        o.trace = trace.data_ptr()
        o.trace_words = trace.numel()
    if workspace is not None:
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    if chunks:
        lib = library()
        arr = (ctypes.c_void_p * D)(*[ctypes.c_void_p(s.data_ptr()) for s in shards])
        st = lib.ag_chunked_matmul_ex(
            arr, D, m, K, ctypes.c_void_p(b.data_ptr()), N,
            ctypes.c_void_p(bias.data_ptr()) if bias is not None else None,
            ctypes.c_void_p(a_gathered.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            _stream_handle(stream), ctypes.byref(o), chunks)
        if st != 0:
            raise AgmmError(st, "ag_chunked_matmul")
        return a_gathered, out
    st = ag_matmul_raw(fused, [s.data_ptr() for s in shards], D, m, K, b.data_ptr(), N,
                       bias.data_ptr() if bias is not None else 0, a_gathered.data_ptr(),
                       out.data_ptr(), _stream_handle(stream), o)
    if st != 0:
        raise AgmmError(st, "ag_matmul" if fused else "ag_then_matmul")
    return a_gathered, out


def ag_matmul(shards, b, bias=None, *, a_gathered=None, out=None, stream=None,
              layout: str = "k_contiguous", rank: int = 0, k_per_flag: int = 0,
              num_sms: int = 0, timeout_ns: int = 0, inject_skip_flag: int = -1, trace=None,
              workspace=None, scale_a: float = 1.0, scale_b: float = 1.0,
              inject_delay_ns: int = 0, **tile):
    """Fused all-gather matmul (one persistent kernel).  Returns (a_gathered, out).
    ``scale_a``/``scale_b``: FP8 per-tensor scales (ignored for 16-bit inputs).
    ``inject_delay_ns``: stress testing, publishers of ready flags wait up to
    this long before publishing.  ``tile``: block_m, block_n, block_k, stages,
    producer_warps (ag_options; 0 = automatic)."""
    return _call(True, shards, b, bias, a_gathered, out, stream, layout, rank, k_per_flag,
                 num_sms, timeout_ns, inject_skip_flag, trace, workspace,
                 scale_a=scale_a, scale_b=scale_b, inject_delay_ns=inject_delay_ns, tile=tile)


def ag_then_matmul(shards, b, bias=None, *, a_gathered=None, out=None, stream=None,
                   layout: str = "k_contiguous", k_per_flag: int = 0, num_sms: int = 0,
                   timeout_ns: int = 0, trace=None, scale_a: float = 1.0, scale_b: float = 1.0,
                   **tile):
    """Barrier baseline: gather kernel, then GEMM kernel.  Returns (a_gathered, out)."""
    return _call(False, shards, b, bias, a_gathered, out, stream, layout, 0, k_per_flag,
                 num_sms, timeout_ns, -1, trace, None, scale_a=scale_a, scale_b=scale_b,
                 tile=tile)


def ag_chunked_matmul(shards, b, bias=None, *, chunks: int = 4, a_gathered=None, out=None,
                      stream=None, num_sms: int = 0, timeout_ns: int = 0, scale_a: float = 1.0,
                      scale_b: float = 1.0):
    """Chunked pipeline: chunk s = the s-th sub-block of every shard; per chunk
    (four streams round-robin) gather it, then multiply its rows.  Returns
    (a_gathered, out); bitwise equal to ag_then_matmul's."""
    if chunks < 1:
        raise ValueError("chunks must be >= 1")
    return _call(False, shards, b, bias, a_gathered, out, stream, "k_contiguous", 0, 0,
                 num_sms, timeout_ns, -1, None, None, chunks=chunks, scale_a=scale_a,
                 scale_b=scale_b)


def device_error(stream=None):
    """Synchronise the stream; return (code, info) of the newest unreported device error."""
    code, info = ctypes.c_int(0), ctypes.c_int(0)
    st = library().ag_get_device_error(_stream_handle(stream), ctypes.byref(code),
                                       ctypes.byref(info))
    if st != 0:
        raise AgmmError(st, "ag_get_device_error")
    return code.value, info.value


def workspace_size(D, m_per_shard, K, N, layout: str = "k_contiguous", k_per_flag: int = 0,
                   dtype: str = "bf16") -> int:
    o = default_options()
    o.layout = LAYOUTS[layout]
    o.k_per_flag = k_per_flag
    o.dtype = DTYPES[dtype]
    return int(library().ag_workspace_size(D, m_per_shard, K, N, ctypes.byref(o)))


def release_workspace() -> None:
    st = library().ag_release_workspace()
    if st != 0:
        raise AgmmError(st, "ag_release_workspace")


class AgPlan(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int32), ("cta_pairs", ctypes.c_int32),
                ("tiles", ctypes.c_int32), ("k_per_flag", ctypes.c_int32),
                ("prologue_cta0", ctypes.c_int32), ("l2_prefetch", ctypes.c_int32),
                ("block_m", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("k_ascending", ctypes.c_int32)]


def plan_fused(D, m_per_shard, K, N, sms, pair_clusters, layout: str = "k_contiguous",
               dtype: str = "bf16", rank: int = 0, k_per_flag: int = 0, num_sms: int = 0,
               **tile) -> dict:
    """The launch plan of a fused call (ag_plan_fused): host arithmetic, no GPU needed."""
    o = default_options()
    o.layout = LAYOUTS[layout]
    o.dtype = DTYPES[dtype]
    o.rank = rank
    o.k_per_flag = k_per_flag
    o.num_sms = num_sms
    for name, value in tile.items():
        if name not in TILE_OPTIONS:
            raise TypeError(f"unknown tile option {name!r}; one of {TILE_OPTIONS}")
        setattr(o, name, value)
    plan = AgPlan()
    st = library().ag_plan_fused(D, m_per_shard, K, N, ctypes.byref(o), sms, pair_clusters,
                                 ctypes.byref(plan))
    if st != 0:
        raise AgmmError(st, "ag_plan_fused")
    return {name: int(getattr(plan, name)) for name, _ in AgPlan._fields_}


def num_sms() -> int:
    return int(library().ag_num_sms())
