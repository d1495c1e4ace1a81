"""GPU tests of the boundary's contract beyond parity: overlap detection on the
library workspace (AG_ERR_BUSY), the delayed-publisher stress run
(inject_delay_ns), the tile options (128-row tiles on single CTAs), and the
bounds-checked build (libagmm_debug.so) on the edge cases.

The ready-flag protocol is the one of "Fused all-gather+GEMM HBM-buffer
kernel for iris.ops" (ROCm/iris #346, description: GEMM workers spin on
per-tile flags that fetchers publish after staging A tiles); the stress run
makes publishers late and out of order so that a reader that does not wait
for a flag, or reads the staged data before the release, returns wrong rows.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import all_gather_gemm_gb300 as agmm
from all_gather_gemm_gb300 import inputs as inp

pytestmark = pytest.mark.gpu

BUSY = 7
REL, ATOL = 1e-2, 1e-3
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    agmm.library()
    yield


def to_device(x):
    return ([s.cuda() for s in x.shards], x.b.cuda(),
            x.bias.cuda() if x.bias is not None else None)


def bits_equal(t1, t2):
    return torch.equal(t1.view(torch.int16), t2.view(torch.int16))


# ---------------------------------------------------------------- AG_ERR_BUSY

def test_busy_when_the_library_workspace_is_in_use_on_another_stream():
    """A fused call on stream s1 that has not run yet (it waits behind a
    spin kernel) holds the library workspace: the same call from s2 returns
    AG_ERR_BUSY and enqueues nothing; so does the m-contiguous barrier call
    (its [K, M] staging is library-owned).  Calls that do not touch the
    library workspace -- the k-contiguous barrier path, a fused call with a
    caller workspace -- and further calls on s1 itself are accepted.  Once s1
    has finished, s2 may use the workspace."""
    w = inp.Workload("busy", D=4, m_per_shard=512, K=1024, N=768, dtype="bf16", bias=True)
    x = inp.make_inputs(w)
    shards, b, bias = to_device(x)
    ref_a, ref_o = agmm.ag_matmul(shards, b, bias)
    ref_bo = agmm.ag_then_matmul(shards, b, bias)[1]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [torch.full_like(ref_o, float("nan")) for _ in range(5)]
    ags = [torch.empty_like(ref_a) for _ in range(5)]
    ws = torch.zeros(agmm.workspace_size(w.D, w.m_per_shard, w.K, w.N), dtype=torch.uint8,
                     device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        torch.cuda._sleep(200_000_000)  # about 0.1 s of spinning ahead of the call
    agmm.ag_matmul(shards, b, bias, a_gathered=ags[0], out=outs[0], stream=s1)
    with pytest.raises(agmm.AgmmError) as e:
        agmm.ag_matmul(shards, b, bias, a_gathered=ags[1], out=outs[1], stream=s2)
    assert e.value.status == BUSY
    with pytest.raises(agmm.AgmmError) as e:
        agmm.ag_then_matmul(shards, b, bias, a_gathered=ags[1], out=outs[1], stream=s2,
                            layout="m_contiguous")
    assert e.value.status == BUSY
    agmm.ag_then_matmul(shards, b, bias, a_gathered=ags[2], out=outs[2], stream=s2)
    agmm.ag_matmul(shards, b, bias, a_gathered=ags[3], out=outs[3], stream=s2, workspace=ws)
    agmm.ag_matmul(shards, b, bias, a_gathered=ags[4], out=outs[4], stream=s1)
    s1.synchronize()
    s2.synchronize()
    assert torch.isnan(outs[1].float()).all(), "a refused call must enqueue nothing"
    agmm.ag_matmul(shards, b, bias, a_gathered=ags[1], out=outs[1], stream=s2)
    s2.synchronize()
    assert agmm.device_error() == (0, 0)
    for i in (0, 1, 3, 4):
        assert bits_equal(outs[i], ref_o), f"call {i}"
        assert bits_equal(ags[i], ref_a), f"call {i} a_gathered"
    assert bits_equal(outs[2], ref_bo)


# ---------------------------------------------------------------- late publishers

STRESS = [
    # (name, workload, layout): a fused call of several waves on each publish path
    ("cube_3200", inp.cube(3200), "k_contiguous"),          # fetch prologue publishes
    ("m4096_d8_k", inp.Workload("m4096_d8", D=8, m_per_shard=512, K=8192, N=3584,
                                dtype="bf16", a_dist="uniform", b_dist="uniform",
                                bias=True), "k_contiguous"),  # owners' copiers, take-overs
    ("m4096_d8_bias_m", inp.iris_m4096_bias(), "m_contiguous"),  # every chunk via [K, M]
    # twelve waves, m-contiguous: k ascending, and pairs wholly in the (rotating) local
    # shard read it directly while every other chunk goes through the [K, M] staging
    ("m16384_d8_m", inp.iris_m16384(), "m_contiguous"),
    ("regfetch", inp.Workload("stress_regfetch", D=5, m_per_shard=130, K=2048, N=1280,
                              dtype="fp16", bias=True), "k_contiguous"),  # register fetcher
]
STRESS_REPS = 50
STRESS_DELAY_NS = 20_000


@pytest.mark.parametrize("name,w,layout", STRESS, ids=[c[0] for c in STRESS])
def test_late_publishers_give_identical_results(name, w, layout):
    """50 fused calls with every publisher waiting a pseudo-random 0-20 us
    before its release store (a different draw each call, since the draw
    hashes the call's epoch), a_gathered and out poisoned before each call and
    the local rank rotating: each result is bitwise the undelayed call's, and
    no wait times out."""
    x = inp.make_inputs(w)
    shards, b, bias = to_device(x)
    ref_a, ref_o = agmm.ag_matmul(shards, b, bias, layout=layout)
    ref_a, ref_o = ref_a.clone(), ref_o.clone()
    assert agmm.device_error() == (0, 0)
    a_g, out = torch.empty_like(ref_a), torch.empty_like(ref_o)
    bad = []
    for rep in range(STRESS_REPS):
        a_g.view(torch.int16).fill_(0x7E00 + rep)  # a NaN pattern in bf16 and fp16
        out.view(torch.int16).fill_(0x7E00 + rep)
        agmm.ag_matmul(shards, b, bias, a_gathered=a_g, out=out, layout=layout,
                       rank=rep % w.D, inject_delay_ns=STRESS_DELAY_NS)
        if not (bits_equal(out, ref_o) and bits_equal(a_g, ref_a)):
            bad.append(rep)
    assert agmm.device_error() == (0, 0)
    assert not bad, f"{name}: results differ from the undelayed call in reps {bad}"


# ---------------------------------------------------------------- tile options

@pytest.mark.parametrize("name,layout", [("m4096_bias", "m_contiguous"),
                                         ("m4096_bias", "k_contiguous"),
                                         ("cube_2432", "k_contiguous")])
def test_single_cta_tiles_on_every_sm(oracle_mod, name, layout):
    """block_m = 128 (one CTA per 128 x 256 tile, 4 stages) on every SM, fused
    and barrier, against the oracle in full; cube_2432 then takes 1.25 waves
    and runs the fetch prologue on single CTAs."""
    w = {"m4096_bias": inp.iris_m4096_bias(), "cube_2432": inp.cube(2432)}[name]
    if name == "cube_2432":
        plan = agmm.plan_fused(w.D, w.m_per_shard, w.K, w.N, agmm.num_sms(), 1, block_m=128)
        assert plan["cta_pairs"] == 0 and plan["prologue_cta0"] >= 0
    x = inp.make_inputs(w)
    shards, b, bias = to_device(x)
    a_f, o_f = agmm.ag_matmul(shards, b, bias, layout=layout, block_m=128, rank=3)
    a_b, o_b = agmm.ag_then_matmul(shards, b, bias, layout=layout, stages=4)
    torch.cuda.synchronize()
    assert agmm.device_error() == (0, 0)
    exp_a = oracle_mod.all_gather(x.shard_bits())
    ref32, _, absab, _ = oracle_mod.gemm_rows(exp_a, x.b_bits(), x.bias_np(), dtype=w.dtype)
    for a_d, o_d, label in ((a_f, o_f, "fused"), (a_b, o_b, "barrier")):
        got_a = a_d.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got_a, exp_a), f"{label}: a_gathered"
        ok, ratio, idx = oracle_mod.within_tolerance(o_d.float().cpu().numpy(), ref32, absab,
                                                     REL, ATOL)
        assert ok, f"{label}: out outside tolerance at {idx} (err/bound {ratio:.3g})"


def test_unsupported_tile_options_enqueue_nothing():
    w = inp.Workload("tile_rej", D=2, m_per_shard=128, K=256, N=256, dtype="bf16")
    x = inp.make_inputs(w)
    shards, b, _ = to_device(x)
    out = torch.full((w.M, w.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    for kw in ({"block_m": 64}, {"stages": 5}, {"block_n": 128}, {"num_sms": 1, "block_m": 256}):
        for fn in (agmm.ag_matmul, agmm.ag_then_matmul):
            with pytest.raises(agmm.AgmmError) as e:
                fn(shards, b, out=out, **kw)
            assert e.value.status == 2, (fn.__name__, kw)
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()


# ---------------------------------------------------------------- bounds-checked build

DEBUG_CASES = [
    "test_gpu_parity.py::test_ragged_shapes",
    "test_gpu_parity.py::test_fetch_prologue",
    "test_gpu_parity.py::test_small_grids_and_flag_granularity",
    "test_gpu_parity.py::test_small_two_shard",
    "test_gpu_fp8.py::test_fp8_ragged",
]


def test_bounds_checked_build_runs_the_edge_cases_clean():
    """libagmm_debug.so checks every flag, per-tile word, shard-row and staging
    index against its buffer on the device and records AG_ERR_BOUNDS instead
    of making the access.  The ragged shapes (D = 16 included), the fetch
    prologue and the small grids run in a fresh process with that build: every
    result matches the oracle and every call reports no device error (the
    parity tests assert device_error() == (0, 0) after each call)."""
    env = dict(os.environ, AGMM_VARIANT="debug")
    probe = subprocess.run(
        [sys.executable, "-c",
         "import all_gather_gemm_gb300 as a; print(a.library()._name)"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert probe.returncode == 0, probe.stderr[-2000:]
    assert probe.stdout.strip().endswith("libagmm_debug.so"), probe.stdout
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
         *[os.path.join(HERE, c) for c in DEBUG_CASES]],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
