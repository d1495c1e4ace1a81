"""ag_matmul_noalloc: the entry point for callers that cannot allocate.

Some callers of this library must not allocate device memory while they run
-- a framework that plans and owns every device allocation up front, or a
latency-critical loop that cannot afford an allocation's implicit device
synchronisation.  ag_matmul may allocate (its error word and flag workspace
on first use, a bigger workspace for a bigger problem); ag_matmul_noalloc
runs the same fused kernel with its scratch in a fixed device array inside
the library instead.  These tests call it through the C ABI and check its
output against ag_matmul_ex's on two calls in a row (the scratch keeps the
previous call's contents, which must not matter), and that it rejects what
its fixed scratch cannot hold.  The file is named to be collected last.
"""
import ctypes

import pytest
import torch

import all_gather_gemm_gb300 as agmm
from all_gather_gemm_gb300 import inputs as inp

pytestmark = pytest.mark.gpu

REL, ATOL = 1e-2, 1e-3  # the parity bound the other GPU tests use
INVALID, UNSUPPORTED, TOO_LARGE = 1, 2, 6


def _noalloc(shards, b, bias, a_g, out, opt):
    lib = agmm.library()
    D = len(shards)
    m, K = shards[0].shape
    N = b.shape[1]
    arr = (ctypes.c_void_p * D)(*[ctypes.c_void_p(s.data_ptr()) for s in shards])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ag_matmul_noalloc(arr, D, m, K, ctypes.c_void_p(b.data_ptr()), N,
                                 ctypes.c_void_p(bias.data_ptr()) if bias is not None else None,
                                 ctypes.c_void_p(a_g.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                 stream, ctypes.byref(opt))


def _within(x, y, a, b):
    """|x - y| <= REL * (|a| @ |b|) + ATOL elementwise, with a = gathered A."""
    scale = a.abs().float() @ b.abs().float()
    return bool(((x.float() - y.float()).abs() <= REL * scale + ATOL).all())


def test_noalloc_matches_ag_matmul_on_two_calls_in_a_row():
    assert torch.cuda.is_available(), "GPU test needs CUDA"
    ws = [inp.Workload("noalloc_a", D=4, m_per_shard=256, K=1024, N=768, dtype="fp16", bias=True),
          inp.Workload("noalloc_b", D=4, m_per_shard=256, K=1024, N=768, dtype="fp16",
                       a_dist="uniform", b_dist="uniform", bias=True, seed=7)]
    results = []
    for w in ws:  # two calls in a row on the shared scratch, different inputs
        x = inp.make_inputs(w)
        shards = [s.cuda() for s in x.shards]
        b, bias = x.b.cuda(), x.bias.cuda()
        a_g = torch.empty(w.M, w.K, dtype=b.dtype, device="cuda")
        out = torch.empty(w.M, w.N, dtype=b.dtype, device="cuda")
        opt = agmm.default_options()
        opt.dtype, opt.rank = 1, 2
        assert _noalloc(shards, b, bias, a_g, out, opt) == 0
        torch.cuda.synchronize()
        results.append((shards, b, bias, a_g.clone(), out.clone()))
    assert agmm.device_error() == (0, 0)
    for shards, b, bias, a_g, out in results:
        ref_a, ref_out = agmm.ag_matmul(shards, b, bias, rank=2)  # the existing entry point
        assert agmm.device_error() == (0, 0)
        assert torch.equal(a_g, torch.cat(shards)) and torch.equal(a_g, ref_a)
        assert _within(out, ref_out, ref_a, b)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))


def test_noalloc_rejects_what_its_scratch_cannot_hold():
    # Rejected before any CUDA call, so well-aligned placeholder addresses do.
    base = 0x7F0000000000
    lib = agmm.library()
    D, m, K, N = 16, 4096, 8192, 3584
    arr = (ctypes.c_void_p * D)(*[ctypes.c_void_p(base + (r << 28)) for r in range(D)])
    args = [arr, D, m, K, ctypes.c_void_p(base + (20 << 28)), N, None,
            ctypes.c_void_p(base + (40 << 28)), ctypes.c_void_p(base + (80 << 28)), None]
    opt = agmm.default_options()
    opt.k_per_flag = 1  # 512 row blocks x 128 flags x 8 bytes: well past 256 KB
    assert lib.ag_matmul_noalloc(*args, ctypes.byref(opt)) == TOO_LARGE
    assert agmm.workspace_size(D, m, K, N, k_per_flag=1) + 256 > 256 * 1024
    opt = agmm.default_options()
    opt.layout = 1
    assert lib.ag_matmul_noalloc(*args, ctypes.byref(opt)) == UNSUPPORTED
    opt = agmm.default_options()
    opt.workspace, opt.workspace_bytes = base + (120 << 28), 1 << 20
    assert lib.ag_matmul_noalloc(*args, ctypes.byref(opt)) == INVALID
    assert lib.ag_status_string(TOO_LARGE)


def test_noalloc_device_timeout_is_reported():
    """A chunk whose ready flag is never published (fault injection, host-set)
    makes a reader's bounded wait run out; the error recorded in the no-alloc
    scratch comes back through ag_get_device_error, and the next call is
    correct again.  Three column blocks give the chunk two readers besides its
    owner, so one of them waits even if the other takes the chunk over."""
    w = inp.Workload("noalloc_inject", D=2, m_per_shard=128, K=256, N=768, dtype="bf16")
    x = inp.make_inputs(w)
    shards = [s.cuda() for s in x.shards]
    b = x.b.cuda()
    a_g = torch.empty(w.M, w.K, dtype=b.dtype, device="cuda")
    out = torch.empty(w.M, w.N, dtype=b.dtype, device="cuda")
    agmm.device_error()  # clear anything older
    opt = agmm.default_options()
    opt.rank, opt.inject_skip_flag, opt.timeout_ns = 1, 0, 20_000_000
    assert _noalloc(shards, b, None, a_g, out, opt) == 0
    assert agmm.device_error() == (4, 0)
    opt = agmm.default_options()
    opt.rank = 1
    assert _noalloc(shards, b, None, a_g, out, opt) == 0
    assert agmm.device_error() == (0, 0)
    ref_a, ref_out = agmm.ag_matmul(shards, b, rank=1)
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))


def test_noalloc_fp8_matches_ag_matmul():
    """FP8 E4M3 (b given as [N, K], bf16 out) through the no-alloc entry: the
    same fused kernel as ag_matmul, so the results are bitwise equal."""
    w = inp.Workload("noalloc_fp8", D=4, m_per_shard=256, K=1024, N=768, dtype="fp8_e4m3",
                     b_scale="one", bias=True, scale_b=0.03)
    x = inp.make_inputs(w)
    shards = [s.cuda() for s in x.shards]
    bt, bias = x.b.cuda(), x.bias.cuda()
    a_g = torch.empty(w.M, w.K, dtype=bt.dtype, device="cuda")
    out = torch.empty(w.M, w.N, dtype=torch.bfloat16, device="cuda")
    opt = agmm.default_options()
    opt.dtype, opt.rank = agmm.DTYPES["fp8_e4m3"], 1
    opt.scale_a, opt.scale_b = w.scale_a, w.scale_b
    lib = agmm.library()
    arr = (ctypes.c_void_p * w.D)(*[ctypes.c_void_p(s.data_ptr()) for s in shards])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.ag_matmul_noalloc(arr, w.D, w.m_per_shard, w.K, ctypes.c_void_p(bt.data_ptr()),
                                 w.N, ctypes.c_void_p(bias.data_ptr()),
                                 ctypes.c_void_p(a_g.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                 stream, ctypes.byref(opt)) == 0
    assert agmm.device_error() == (0, 0)
    ref_a, ref_out = agmm.ag_matmul(shards, bt, bias, rank=1, scale_a=w.scale_a,
                                    scale_b=w.scale_b)
    assert agmm.device_error() == (0, 0)
    assert torch.equal(a_g.view(torch.uint8), ref_a.view(torch.uint8))
    assert torch.equal(out, ref_out)


@pytest.mark.parametrize("name", ["multi_wave", "fetch_prologue"])
def test_noalloc_multi_wave_and_prologue_match_ag_matmul(name):
    """Calls of more than one wave on the shared scratch: M=4096 N=3584
    K=8192 over 8 shards takes three waves of CTA pairs, where per-tile words
    left by the previous call decide between waiting for a chunk's owner and
    taking the chunk over; cube 2432 takes 1.3 waves and its CTAs with a tile
    fewer first stage all of A (the fetch prologue).  Two calls in a row each,
    bitwise equal to ag_matmul (the same kernel and launch plan)."""
    w = {"multi_wave": inp.Workload("noalloc_mw", D=8, m_per_shard=512, K=8192, N=3584,
                                    dtype="bf16", bias=True),
         "fetch_prologue": inp.cube(2432)}[name]
    sms = agmm.num_sms()
    plan = agmm.plan_fused(w.D, w.m_per_shard, w.K, w.N, sms, sms // 2)
    assert plan["tiles"] > plan["grid"] // 2
    if name == "fetch_prologue":
        assert plan["prologue_cta0"] >= 0
    x = inp.make_inputs(w)
    shards = [s.cuda() for s in x.shards]
    b = x.b.cuda()
    bias = x.bias.cuda() if x.bias is not None else None
    ref_a, ref_out = agmm.ag_matmul(shards, b, bias, rank=1)
    ref_a, ref_out = ref_a.clone(), ref_out.clone()
    assert agmm.device_error() == (0, 0)
    for call in range(2):
        a_g = torch.full_like(ref_a, float("nan"))
        out = torch.full_like(ref_out, float("nan"))
        opt = agmm.default_options()
        opt.rank = 1
        assert _noalloc(shards, b, bias, a_g, out, opt) == 0
        assert agmm.device_error() == (0, 0)
        assert torch.equal(a_g.view(torch.int16), ref_a.view(torch.int16)), f"call {call}"
        assert _within(out, ref_out, ref_a, b)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"call {call}"
