"""The C-ABI boundary on the CPU: the library builds, loads, exports every
function include/agmm.h declares, and rejects bad arguments with the
documented status before touching CUDA (no GPU needed)."""
import ctypes
import os
import re

import pytest

import all_gather_gemm_gb300 as agmm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "agmm.h")

INVALID, UNSUPPORTED, CUDA, WORKSPACE = 1, 2, 3, 5


@pytest.fixture(scope="module")
def lib():
    return agmm.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(ag_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    assert set(agmm.EXPORTS) <= set(names), names
    assert {"ag_matmul", "ag_then_matmul"} <= set(names)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_options_default_matches_header(lib):
    o = agmm.AgOptions()
    ctypes.memset(ctypes.byref(o), 0x5A, ctypes.sizeof(o))
    lib.ag_options_default(ctypes.byref(o))
    assert (o.dtype, o.layout, o.rank, o.k_per_flag, o.num_sms) == (0, 0, 0, 0, 0)
    assert o.inject_skip_flag == -1 and o.timeout_ns == 2_000_000_000
    assert not o.trace and o.trace_words == 0 and not o.workspace and o.workspace_bytes == 0
    assert o.scale_a == 1.0 and o.scale_b == 1.0
    assert o.inject_delay_ns == 0
    assert (o.block_m, o.block_n, o.block_k, o.stages, o.producer_warps) == (0, 0, 0, 0, 0)
    assert ctypes.sizeof(o) == 104


def test_status_strings(lib):
    unknown = lib.ag_status_string(99)
    assert unknown == b"unknown status"
    for code in range(9):
        s = lib.ag_status_string(code)
        assert isinstance(s, bytes) and s and s != unknown, code
    assert b"busy" in lib.ag_status_string(7) or b"in use" in lib.ag_status_string(7)
    assert b"bounds" in lib.ag_status_string(8) or b"outside" in lib.ag_status_string(8)
    assert set(agmm.STATUS) == set(range(9))


def test_workspace_size(lib):
    # automatic k_per_flag is sized at its finest, 4 k-blocks per flag:
    # flags: 8 row blocks x (128 k-blocks / 4 per flag) x 8 bytes = 2 KiB;
    # started words: (8 + 1) x 14 tile slots x 8 bytes = 1008 B -> 1 KiB
    assert agmm.workspace_size(8, 128, 8192, 3584) == 2048 + 1024
    # 128 row blocks x 32 flags x 8 bytes = 32 KiB, (128 + 1) x 14 tile slots x 8 B
    # = 14448 B -> 15 KiB, plus [K, M] staging for m-contiguous
    assert agmm.workspace_size(8, 2048, 8192, 3584) == 32768 + 15360
    assert agmm.workspace_size(8, 2048, 8192, 3584, "m_contiguous") == (
        32768 + 15360 + 16384 * 8192 * 2)
    assert agmm.workspace_size(8, 2048, 8192, 3584, k_per_flag=1) == 128 * 128 * 8 + 15360
    assert agmm.workspace_size(8, 2048, 8192, 3584, k_per_flag=16) == 8192 + 15360
    assert agmm.workspace_size(1, 1, 8, 8) == 2048  # one flag and one tile, 1 KiB each
    # automatic granularity, sized at 4 k-blocks per flag: K=384 has 6 k-blocks
    # -> 2 flags per row block (3 row blocks): 48 B -> 1 KiB
    assert agmm.workspace_size(8, 48, 384, 384) == 1024 + 1024
    # FP8 (8-bit elements) is sized like the 16-bit problem with K/2 columns;
    # K must be a multiple of 16 (16-byte rows)
    assert agmm.workspace_size(8, 2048, 16384, 3584, dtype="fp8_e4m3") == 32768 + 15360
    assert agmm.workspace_size(8, 2048, 8200, 3584, dtype="fp8_e4m3") == 0
    assert agmm.workspace_size(8, 48, 384, 384, k_per_flag=8) == 1024 + 1024
    assert agmm.workspace_size(0, 1, 8, 8) == 0
    assert agmm.workspace_size(1, 1, 12, 8) == 0


# Fake, well-aligned, non-overlapping "device" addresses: validation rejects
# these calls before any CUDA call, so nothing is ever dereferenced.
BASE = 0x7F0000000000


def _call(lib, fused=True, D=2, m=128, K=256, N=256, shards=None, b=BASE + (1 << 30),
          bias=None, ag=BASE + (2 << 30), out=BASE + (3 << 30), opt=None):
    if shards is None:
        shards = [BASE + (r << 24) for r in range(D)]
    return agmm.ag_matmul_raw(fused, shards, D, m, K, b, N, bias, ag, out, None, opt)


def opts(**kw):
    o = agmm.default_options()
    for k, v in kw.items():
        setattr(o, k, v)
    return o


@pytest.mark.parametrize("fused", [True, False])
def test_invalid_arguments_are_rejected_before_cuda(lib, fused):
    assert _call(lib, fused, b=0) == INVALID
    assert _call(lib, fused, ag=0) == INVALID
    assert _call(lib, fused, out=0) == INVALID
    assert _call(lib, fused, shards=[BASE, 0]) == INVALID
    assert _call(lib, fused, D=0, shards=[]) == INVALID
    assert _call(lib, fused, m=0) == INVALID
    assert _call(lib, fused, K=0) == INVALID
    assert _call(lib, fused, K=250) == INVALID           # K % 8
    assert _call(lib, fused, N=12) == INVALID            # N % 8
    assert _call(lib, fused, b=BASE + (1 << 30) + 8) == INVALID   # not 16-byte aligned
    assert _call(lib, fused, shards=[BASE + 4, BASE + (1 << 24)]) == INVALID
    assert _call(lib, fused, bias=BASE + (4 << 30) + 2) == INVALID  # bias not 4-byte aligned
    # outputs overlapping inputs or each other
    assert _call(lib, fused, out=BASE + (2 << 30) + 4096) == INVALID
    assert _call(lib, fused, ag=BASE + 1024) == INVALID
    assert _call(lib, fused, out=BASE + (1 << 30)) == INVALID
    assert _call(lib, fused, opt=opts(rank=2)) == INVALID
    assert _call(lib, fused, opt=opts(rank=-1)) == INVALID
    assert _call(lib, fused, opt=opts(dtype=7)) == INVALID
    assert _call(lib, fused, opt=opts(layout=3)) == INVALID
    assert _call(lib, fused, opt=opts(timeout_ns=-5)) == INVALID
    assert _call(lib, fused, opt=opts(k_per_flag=-1)) == INVALID
    D = 17  # one more than AG_MAX_SHARDS
    assert _call(lib, fused, D=D, m=1, shards=[BASE + (r << 24) for r in range(D)]) == UNSUPPORTED
    assert _call(lib, fused, opt=opts(k_per_flag=65537)) == INVALID


@pytest.mark.parametrize("fused", [True, False])
def test_tile_options_accept_only_compiled_shapes(lib, fused):
    """block_m / block_n / block_k / stages / producer_warps: the pages'
    tunables; only the compiled shapes pass validation (a valid one then
    reaches the first CUDA call, CUDA or UNSUPPORTED without a GPU)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("this check is for hosts without a GPU")
    for kw in ({"block_m": 64}, {"block_m": 512}, {"block_n": 128}, {"block_k": 32},
               {"block_k": 128}, {"stages": 5}, {"stages": 8}, {"producer_warps": 8},
               {"block_m": 128, "stages": 6}, {"block_m": 256, "stages": 4}):
        assert _call(lib, fused, opt=opts(**kw)) == UNSUPPORTED, kw
    for kw in ({"block_m": -1}, {"block_n": -256}, {"block_k": -64}, {"stages": -6},
               {"producer_warps": -4}):
        assert _call(lib, fused, opt=opts(**kw)) == INVALID, kw
    for kw in ({"block_m": 128}, {"block_m": 256}, {"block_n": 256}, {"block_k": 64},
               {"stages": 4}, {"stages": 6}, {"producer_warps": 4},
               {"block_m": 256, "block_n": 256, "block_k": 64, "stages": 6, "producer_warps": 4}):
        assert _call(lib, fused, opt=opts(**kw)) in (CUDA, UNSUPPORTED), kw
    # FP8 counts block_k in 8-bit elements: 128 per stage
    assert _call(lib, fused, opt=opts(dtype=2, block_k=64)) == UNSUPPORTED
    assert _call(lib, fused, opt=opts(dtype=2, block_k=128)) in (CUDA, UNSUPPORTED)


@pytest.mark.parametrize("fused", [True, False])
def test_inject_delay_is_bounded_by_the_timeout(lib, fused):
    import torch
    if torch.cuda.is_available():
        pytest.skip("this check is for hosts without a GPU")
    assert _call(lib, fused, opt=opts(inject_delay_ns=-1)) == INVALID
    # at most timeout_ns / 16: 125 ms with the default 2 s
    assert _call(lib, fused, opt=opts(inject_delay_ns=125_000_001)) == INVALID
    assert _call(lib, fused, opt=opts(inject_delay_ns=125_000_000)) in (CUDA, UNSUPPORTED)
    assert _call(lib, fused, opt=opts(timeout_ns=16_000, inject_delay_ns=1001)) == INVALID
    assert _call(lib, fused, opt=opts(timeout_ns=16_000, inject_delay_ns=1000)) in (CUDA,
                                                                                   UNSUPPORTED)


@pytest.mark.parametrize("fused", [True, False])
def test_m_contiguous_needs_m_multiple_of_8(lib, fused):
    assert _call(lib, fused, D=3, m=3, opt=opts(layout=1)) == UNSUPPORTED


def _chunked(lib, chunks, opt=None, D=2, m=128, K=256, N=256, b=BASE + (1 << 30)):
    arr = (ctypes.c_void_p * D)(*[ctypes.c_void_p(BASE + (r << 24)) for r in range(D)])
    o = opt if opt is not None else agmm.default_options()
    return lib.ag_chunked_matmul_ex(arr, D, m, K, ctypes.c_void_p(b), N, None,
                                    ctypes.c_void_p(BASE + (2 << 30)),
                                    ctypes.c_void_p(BASE + (3 << 30)), None, ctypes.byref(o),
                                    chunks)


def test_chunked_pipeline_arguments_are_checked_before_cuda(lib):
    assert _chunked(lib, 0) == INVALID
    assert _chunked(lib, -3) == INVALID
    assert _chunked(lib, 4097) == INVALID
    assert _chunked(lib, 4, b=0) == INVALID
    assert _chunked(lib, 4, K=250) == INVALID
    assert _chunked(lib, 4, opt=opts(layout=1)) == UNSUPPORTED  # k-contiguous only


def test_valid_call_without_a_gpu_reports_cuda_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("this check is for hosts without a GPU")
    assert _call(lib, True) in (CUDA, UNSUPPORTED)
    assert _call(lib, False) in (CUDA, UNSUPPORTED)
    assert lib.ag_num_sms() == 0
    code, info = ctypes.c_int(-1), ctypes.c_int(-1)
    assert lib.ag_get_device_error(None, ctypes.byref(code), ctypes.byref(info)) == CUDA
    assert code.value == 0


def test_python_binding_fails_loudly_without_cuda_tensors():
    import torch
    s = [torch.zeros(4, 8, dtype=torch.bfloat16)]
    with pytest.raises((ValueError, RuntimeError)):
        agmm.ag_matmul(s, torch.zeros(8, 8, dtype=torch.bfloat16))


def test_library_variant_selection(monkeypatch):
    """AGMM_VARIANT=debug or AGMM_DEBUG=1 select the bounds-checked build;
    anything else unknown is refused."""
    for env, want in (({}, "release"), ({"AGMM_DEBUG": "1"}, "debug"),
                      ({"AGMM_DEBUG": "0"}, "release"), ({"AGMM_VARIANT": "debug"}, "debug"),
                      ({"AGMM_VARIANT": "release", "AGMM_DEBUG": "1"}, "release")):
        monkeypatch.delenv("AGMM_VARIANT", raising=False)
        monkeypatch.delenv("AGMM_DEBUG", raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        assert agmm.variant() == want, env
    monkeypatch.setenv("AGMM_VARIANT", "fast")
    with pytest.raises(ValueError):
        agmm.variant()
