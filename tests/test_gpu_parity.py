"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

a_gathered must be bit-exact; out must satisfy, elementwise,
    |out_gpu - out_ref_f32| <= 1e-2 * (|a|.|b|)_ij + 1e-3
where out_ref_f32 is the oracle's fp32 sum (+ bias) and (|a|.|b|)_ij the sum
of |a_ik||b_kj|.  Every output element is checked, at every size (the
oracle takes about 6 s for the largest workload, M=16384 N=3584 K=8192, on
the 16 host cores of a GB300 machine).  Both the fused kernel and the barrier
baseline are checked against the oracle.  The fused kernel's k order is fixed per tile, so its
outputs must be bitwise equal for every choice of local rank and staging
layout; the barrier GEMM runs k in ascending order (a different fp32
summation order), so it is bitwise equal to itself across layouts.
"""
import numpy as np
import pytest
import torch

import all_gather_gemm_gb300 as agmm
from all_gather_gemm_gb300 import inputs as inp

pytestmark = pytest.mark.gpu

REL, ATOL = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    agmm.library()
    yield


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def to_device(x: inp.Inputs):
    shards = [s.cuda() for s in x.shards]
    b = x.b.cuda()
    bias = x.bias.cuda() if x.bias is not None else None
    return shards, b, bias


def check(oracle, x: inp.Inputs, a_dev, out_dev, rows=None, what="", more=()):
    """a_gathered bit-exact and out within tolerance of the oracle; `more` =
    further (a, out, label) results of the same inputs, checked against the
    same oracle computation."""
    exp_a = oracle.all_gather(x.shard_bits())
    ref32, _, _abs, _ = oracle.gemm_rows(exp_a, x.b_bits(), x.bias_np(), dtype=x.workload.dtype,
                                         rows=rows)
    ratio = 0.0
    for a_d, o_d, label in ((a_dev, out_dev, what),) + tuple(more):
        got_a = bits(a_d)
        assert np.array_equal(got_a, exp_a), \
            f"{label}: a_gathered differs at {np.argwhere(got_a != exp_a)[:3]}"
        got = o_d if rows is None else o_d[torch.as_tensor(rows, device=o_d.device)]
        got32 = got.float().cpu().numpy()
        ok, r_, idx = oracle.within_tolerance(got32, ref32, _abs, REL, ATOL)
        r = None if idx is None else (int(rows[idx[0]]) if rows is not None else idx[0], idx[1])
        assert ok, f"{label}: out outside tolerance (worst err/bound {r_:.3g}) at (row, col) {r}"
        ratio = max(ratio, r_)
    return ratio


def run_both(x, layout="k_contiguous", rank=0, **kw):
    shards, b, bias = to_device(x)
    a_f, o_f = agmm.ag_matmul(shards, b, bias, layout=layout, rank=rank, **kw)
    a_b, o_b = agmm.ag_then_matmul(shards, b, bias, layout=layout)
    torch.cuda.synchronize()
    code, info = agmm.device_error()
    assert code == 0, f"device error {code} info {info:#x}"
    return (a_f, o_f), (a_b, o_b)


def assert_bitwise(t1, t2, what):
    assert torch.equal(t1.view(torch.int16), t2.view(torch.int16)), what


# ---------------------------------------------------------------- the five workloads

def test_small_two_shard(oracle_mod):
    x = inp.make_inputs(inp.small_two_shard())
    (a_f, o_f), (a_b, o_b) = run_both(x)
    check(oracle_mod, x, a_f, o_f, what="fused", more=((a_b, o_b, "barrier"),))


@pytest.mark.parametrize("n", list(range(256, 4096 + 1, 128)))
def test_cube_sweep(oracle_mod, n):
    w = inp.cube(n)
    x = inp.make_inputs(w)
    (a_f, o_f), (a_b, o_b) = run_both(x)
    check(oracle_mod, x, a_f, o_f, what=f"fused cube {n}",
          more=((a_b, o_b, f"barrier cube {n}"),))


@pytest.mark.parametrize("D", [2, 4, 8])
def test_iris_m1024(oracle_mod, D):
    w = inp.iris_m1024(D)
    x = inp.make_inputs(w)
    (a_f, o_f), (a_b, o_b) = run_both(x)
    check(oracle_mod, x, a_f, o_f, what=f"m1024 D={D}",
          more=((a_b, o_b, f"barrier m1024 D={D}"),))


def test_iris_m16384_both_layouts(oracle_mod):
    w = inp.iris_m16384()
    x = inp.make_inputs(w)
    shards, b, _ = to_device(x)
    a_k, o_k = agmm.ag_matmul(shards, b, layout="k_contiguous")
    a_m, o_m = agmm.ag_matmul(shards, b, layout="m_contiguous")
    a_b, o_b = agmm.ag_then_matmul(shards, b)
    a_bm, o_bm = agmm.ag_then_matmul(shards, b, layout="m_contiguous")
    assert agmm.device_error() == (0, 0)
    check(oracle_mod, x, a_k, o_k, what="k_contiguous",
          more=((a_b, o_b, "barrier k_contiguous"),))
    assert_bitwise(a_m, a_k, "a_gathered m vs k")
    assert_bitwise(o_m, o_k, "out m_contiguous vs k_contiguous")
    assert_bitwise(a_bm, a_k, "a_gathered barrier m")
    assert_bitwise(o_bm, o_b, "out barrier m_contiguous vs barrier k_contiguous")
    # twelve waves: the plan runs every fused tile k ascending, as the barrier GEMM
    sms = agmm.num_sms()
    assert agmm.plan_fused(w.D, w.m_per_shard, w.K, w.N, sms, sms // 2,
                           dtype="fp16")["k_ascending"] == 1
    assert_bitwise(o_k, o_b, "fused (k ascending) vs barrier")


@pytest.mark.parametrize("layout", ["k_contiguous", "m_contiguous"])
def test_output_sharded_slice(oracle_mod, layout):
    """Output-sharded form: one rank's N/8 column slice of the M=16384 problem
    (b column-sharded) through the same entry points; the gather is the full
    one, the GEMM eight times smaller."""
    w = inp.iris_m16384_colshard()
    x = inp.make_inputs(w)
    (a_f, o_f), (a_b, o_b) = run_both(x, layout=layout)
    check(oracle_mod, x, a_f, o_f, what=f"colshard {layout}",
          more=((a_b, o_b, f"barrier colshard {layout}"),))


def test_iris_m4096_bias_m_contiguous(oracle_mod):
    w = inp.iris_m4096_bias()
    x = inp.make_inputs(w)
    (a_f, o_f), (a_b, o_b) = run_both(x, layout="m_contiguous")
    check(oracle_mod, x, a_f, o_f, what="bias m_contiguous",
          more=((a_b, o_b, "barrier bias m_contiguous"),))


# ---------------------------------------------------------------- edge cases

RAGGED = [
    # (D, m_per_shard, K, N, dtype)
    (1, 1, 8, 8, "bf16"),
    (3, 37, 200, 136, "bf16"),
    (2, 64, 1032, 264, "fp16"),
    (5, 130, 72, 520, "bf16"),
    (8, 16, 64, 64, "fp16"),
    (1, 300, 128, 1000, "bf16"),
    (7, 100, 3000, 40, "fp16"),
    (16, 24, 136, 72, "bf16"),   # the maximum shard count; 8-row boxes straddle shards
]


@pytest.mark.parametrize("D,m,K,N,dt", RAGGED)
def test_ragged_shapes(oracle_mod, D, m, K, N, dt):
    w = inp.Workload(f"ragged_{D}_{m}_{K}_{N}", D=D, m_per_shard=m, K=K, N=N, dtype=dt,
                     a_dist="uniform", b_dist="uniform", b_scale="one", bias=(D % 2 == 1))
    x = inp.make_inputs(w)
    for rank in sorted({0, D - 1}):
        (a_f, o_f), (a_b, o_b) = run_both(x, rank=rank)
        check(oracle_mod, x, a_f, o_f, what=f"fused rank {rank}", more=((a_b, o_b, "barrier"),))
        if w.M % 8 == 0:
            (a_m, o_m), (a_bm, o_bm) = run_both(x, layout="m_contiguous", rank=rank)
            assert_bitwise(a_m, a_f, "a_gathered m vs k")
            assert_bitwise(o_m, o_f, "m_contiguous vs k_contiguous")
            assert_bitwise(a_bm, a_f, "barrier a_gathered m vs k")
            assert_bitwise(o_bm, o_b, "barrier m_contiguous vs k_contiguous")


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_integer_inputs_exact(oracle_mod, dt):
    """Integer entries in [-4, 4] and K=256: every partial sum is an exact
    fp32 integer, so the GPU result must equal the oracle bit for bit."""
    g = torch.Generator().manual_seed(5)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    D, m, K, N = 2, 192, 256, 384
    a = torch.randint(-4, 5, (D * m, K), generator=g).to(tdt)
    b = torch.randint(-4, 5, (K, N), generator=g).to(tdt)
    shards = [a[r * m:(r + 1) * m].contiguous().cuda() for r in range(D)]
    a_g, out = agmm.ag_matmul(shards, b.cuda(), rank=1)
    assert agmm.device_error() == (0, 0)
    exact = (a.to(torch.int64) @ b.to(torch.int64)).to(torch.float32).to(tdt)
    assert_bitwise(out.cpu(), exact, "integer GEMM")
    _, _, obits, _ = oracle_mod.ag_matmul([bits(s) for s in shards], bits(b), dtype=dt,
                                          want_abs=False)
    assert np.array_equal(bits(out), obits)


def test_identity_b_returns_gathered_a():
    g = torch.Generator().manual_seed(6)
    D, m, K = 4, 96, 384
    shards = [torch.randn(m, K, generator=g).to(torch.bfloat16).cuda() for _ in range(D)]
    eye = torch.eye(K, dtype=torch.bfloat16, device="cuda")
    a_g, out = agmm.ag_matmul(shards, eye, rank=2)
    assert agmm.device_error() == (0, 0)
    assert_bitwise(out, a_g, "a @ I")
    assert_bitwise(a_g, torch.cat(shards), "a_gathered")


def test_rank_invariance(oracle_mod):
    w = inp.cube(1024)
    x = inp.make_inputs(w)
    shards, b, _ = to_device(x)
    ref_a, ref_o = agmm.ag_matmul(shards, b, rank=0)
    for rank in (1, 3, 7):
        for layout in ("k_contiguous", "m_contiguous"):
            a_r, o_r = agmm.ag_matmul(shards, b, rank=rank, layout=layout)
            assert agmm.device_error() == (0, 0)
            assert_bitwise(a_r, ref_a, f"a_gathered rank {rank} {layout}")
            assert_bitwise(o_r, ref_o, f"out rank {rank} {layout}")
    check(oracle_mod, x, ref_a, ref_o, what="cube 1024 rank 0")


@pytest.mark.parametrize("num_sms,kpf", [(1, 16), (3, 1), (7, 4), (0, 2)])
def test_small_grids_and_flag_granularity(oracle_mod, num_sms, kpf):
    """Few CTAs (or 1) must still complete: a CTA's own fetch warps stage every
    chunk its tiles need, so no CTA waits on a CTA that is not running."""
    w = inp.Workload("grid", D=4, m_per_shard=160, K=1024, N=512, dtype="bf16")
    x = inp.make_inputs(w)
    shards, b, _ = to_device(x)
    for rank in (0, 2):
        a_f, o_f = agmm.ag_matmul(shards, b, rank=rank, num_sms=num_sms, k_per_flag=kpf)
        assert agmm.device_error() == (0, 0)
        check(oracle_mod, x, a_f, o_f, what=f"num_sms={num_sms} kpf={kpf} rank={rank}")


# (D, m_per_shard, K, N, dtype, bias, rank): on 40 SMs (20 CTA pairs) each takes
# between one and three waves with a partial last one, so the CTAs with one
# tile fewer run the fetch prologue; ragged K and N, a half-empty last pair,
# row blocks straddling shards (64- and 8-row boxes) and a non-zero rank.
PROLOGUE = [
    (4, 384, 520, 1024, "bf16", True, 0),
    (8, 200, 256, 776, "fp16", False, 5),
    (2, 704, 136, 1800, "bf16", False, 1),
]


@pytest.mark.parametrize("D,m,K,N,dt,bias,rank", PROLOGUE)
def test_fetch_prologue(oracle_mod, D, m, K, N, dt, bias, rank):
    """Calls with a partial last wave: the CTAs with fewer tiles stage every
    chunk of A before their own tiles (trace role 4, each exactly once), the
    others wait on those flags; results as the oracle (so are those of the
    same call on all SMs: one wave, no prologue) and bitwise equal to the
    barrier path (k ascending in both)."""
    w = inp.Workload(f"prologue_{D}_{m}_{K}_{N}", D=D, m_per_shard=m, K=K, N=N, dtype=dt,
                     a_dist="uniform", b_dist="uniform", bias=bias)
    x = inp.make_inputs(w)
    shards, b, bias_d = to_device(x)
    tr = torch.zeros(1 + 4 * 16384, dtype=torch.int64, device="cuda")
    a_f, o_f = agmm.ag_matmul(shards, b, bias_d, rank=rank, num_sms=40, trace=tr)
    a_b, o_b = agmm.ag_then_matmul(shards, b, bias_d)
    a_1, o_1 = agmm.ag_matmul(shards, b, bias_d, rank=rank)
    torch.cuda.synchronize()
    assert agmm.device_error() == (0, 0)
    t = tr.cpu().numpy().view(np.uint64)
    n = int(t[0])
    assert n <= 16384
    rec = t[1:1 + 4 * n].reshape(-1, 4)
    pro = rec[(rec[:, 2] >> np.uint64(56)) == 4]
    num_mb, num_kb = -(-w.M // 128), -(-K // 64)
    G = -(-num_kb // 8)  # automatic k_per_flag for more than one wave: 8
    keys = sorted((((pro[:, 2] >> np.uint64(20)) & np.uint64(0xFFFFF)) * np.uint64(G)
                   + (pro[:, 2] & np.uint64(0xFFFFF))).tolist())
    assert keys == list(range(num_mb * G)), "every chunk staged once by the prologue"
    check(oracle_mod, x, a_f, o_f, what="fused, fetch prologue",
          more=((a_b, o_b, "barrier"), (a_1, o_1, "fused, all SMs")))
    assert_bitwise(o_f, o_b, "prologue vs barrier")


@pytest.mark.parametrize("num_sms", [1, 2, 3, 7, 0])
@pytest.mark.parametrize("layout", ["k_contiguous", "m_contiguous"])
def test_barrier_small_grids_odd_row_blocks(oracle_mod, num_sms, layout):
    """The barrier GEMM runs on CTA pairs (256-row tiles) when at least two SMs
    are allowed: 5 row blocks leave the last pair half empty, and 1, 2 or 3
    SMs give one CTA, one pair, or one pair plus an idle SM."""
    w = inp.Workload("grid_odd", D=4, m_per_shard=160, K=1024, N=520, dtype="fp16", bias=True)
    x = inp.make_inputs(w)
    shards, b, bias = to_device(x)
    a_b, o_b = agmm.ag_then_matmul(shards, b, bias, layout=layout, num_sms=num_sms)
    assert agmm.device_error() == (0, 0)
    check(oracle_mod, x, a_b, o_b, what=f"barrier num_sms={num_sms} {layout}")


@pytest.mark.parametrize("name,chunks", [("two_shard", 1), ("two_shard", 3), ("ragged", 4),
                                         ("cube_1280", 4), ("m1024_d8", 8), ("m16384_d8", 4),
                                         ("uneven", 3), ("uneven", 64)])
def test_chunked_pipeline(oracle_mod, name, chunks):
    """The chunked pipeline (chunk s = the s-th sub-block of every shard,
    gathered then multiplied, chunks round-robin over four streams) gives
    a_gathered bitwise and the barrier's out bitwise (same GEMM core and k
    order), which the oracle checks in full."""
    w = {"two_shard": inp.small_two_shard(), "cube_1280": inp.cube(1280),
         "m1024_d8": inp.iris_m1024(8), "m16384_d8": inp.iris_m16384(),
         "ragged": inp.Workload("ragged_chunk", D=3, m_per_shard=37, K=200, N=136, dtype="bf16",
                                a_dist="uniform", b_dist="uniform", b_scale="one",
                                bias=True),
         # 640-row shards in 3 (or, capped, 5) chunks: 213/213/214-row sub-blocks,
         # each padded to 2 row blocks
         "uneven": inp.Workload("uneven_chunk", D=3, m_per_shard=640, K=512, N=392,
                                dtype="fp16", bias=True)}[name]
    x = inp.make_inputs(w)
    shards, b, bias = to_device(x)
    a_c, o_c = agmm.ag_chunked_matmul(shards, b, bias, chunks=chunks)
    a_b, o_b = agmm.ag_then_matmul(shards, b, bias)
    torch.cuda.synchronize()
    assert agmm.device_error() == (0, 0)
    assert_bitwise(a_c, a_b, "chunked a_gathered")
    assert_bitwise(o_c, o_b, "chunked out vs barrier")
    check(oracle_mod, x, a_c, o_c, what=f"chunked {name} S={chunks}")


def test_repeat_calls_are_deterministic():
    x = inp.make_inputs(inp.cube(1536))
    shards, b, _ = to_device(x)
    a1, o1 = agmm.ag_matmul(shards, b, rank=5)
    outs = [agmm.ag_matmul(shards, b, rank=5)[1] for _ in range(5)]
    assert agmm.device_error() == (0, 0)
    for o in outs:
        assert_bitwise(o, o1, "repeat")


def test_caller_workspace(oracle_mod):
    w = inp.Workload("ws", D=4, m_per_shard=256, K=512, N=768, dtype="fp16", bias=True)
    x = inp.make_inputs(w)
    shards, b, bias = to_device(x)
    for layout in ("k_contiguous", "m_contiguous"):
        nbytes = agmm.workspace_size(w.D, w.m_per_shard, w.K, w.N, layout)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        ref_a, ref_o = agmm.ag_matmul(shards, b, bias, layout=layout)
        for _ in range(2):
            a_w, o_w = agmm.ag_matmul(shards, b, bias, layout=layout, workspace=ws, rank=1)
            assert agmm.device_error() == (0, 0)
            assert_bitwise(o_w, ref_o, f"workspace {layout}")
            assert_bitwise(a_w, ref_a, f"workspace a {layout}")
        small = torch.zeros(max(nbytes - 1024, 256), dtype=torch.uint8, device="cuda")
        with pytest.raises(agmm.AgmmError) as e:
            agmm.ag_matmul(shards, b, bias, layout=layout, workspace=small)
        assert e.value.status == 5
    check(oracle_mod, x, ref_a, ref_o, what="workspace")


def test_host_pointer_is_rejected():
    s = [torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")]
    b = torch.zeros(64, 64, dtype=torch.bfloat16)  # host memory
    st = agmm.ag_matmul_raw(True, [s[0].data_ptr()], 1, 128, 64, b.data_ptr(), 64, 0,
                            torch.empty(128, 64, dtype=torch.bfloat16, device="cuda").data_ptr(),
                            torch.empty(128, 64, dtype=torch.bfloat16, device="cuda").data_ptr(),
                            None)
    assert st == 1


# ---------------------------------------------------------------- failure detection

def test_ready_flag_timeout_is_reported_and_context_survives(oracle_mod):
    """Fault injection: chunk 0 (row block 0, which lies in the non-local
    shard) is never published, so a reader of that row block runs its bounded
    wait out; the kernel records AG_ERR_TIMEOUT with the flag index, finishes,
    and the next call on the same context is correct.  Three column blocks
    give the chunk an owner and two readers: a reader that finds the owner not
    yet started takes the chunk over (and never publishes it either), which
    leaves the other reader waiting, so the timeout does not depend on timing."""
    w = inp.Workload("inject", D=2, m_per_shard=128, K=256, N=768, dtype="bf16")
    x = inp.make_inputs(w)
    shards, b, _ = to_device(x)
    agmm.device_error()  # clear anything older
    agmm.ag_matmul(shards, b, rank=1, inject_skip_flag=0, timeout_ns=20_000_000)
    code, info = agmm.device_error()
    assert (code, info) == (4, 0)
    a_g, out = agmm.ag_matmul(shards, b, rank=1)
    assert agmm.device_error() == (0, 0)
    check(oracle_mod, x, a_g, out, what="after timeout")


def test_trace_records_overlap_roles():
    w = inp.cube(2048)
    x = inp.make_inputs(w)
    shards, b, _ = to_device(x)
    tr = torch.zeros(1 + 4 * 8192, dtype=torch.int64, device="cuda")
    agmm.ag_matmul(shards, b, rank=0, trace=tr, k_per_flag=4)
    assert agmm.device_error() == (0, 0)
    t = tr.cpu().numpy().view(np.uint64)
    n = int(t[0])
    rec = t[1:1 + 4 * min(n, 8192)].reshape(-1, 4)
    roles = set(int(r) >> 56 for r in rec[:, 2])
    assert {1, 3} <= roles
    assert np.all(rec[:, 1] >= rec[:, 0])
    fetch = rec[(rec[:, 2] >> np.uint64(56)) == 1]
    # every (row block, k-group) chunk is staged by its owner (or a follower
    # that took it over) at least once
    num_mb, G = 2048 // 128, 2048 // 64 // 4  # 32 k-blocks, 4 per flag
    keys = ((fetch[:, 2] >> np.uint64(20)) & np.uint64(0xFFFFF)) * np.uint64(G) + (fetch[:, 2] & np.uint64(0xFFFFF))
    assert set(keys.tolist()) == set(range(num_mb * G))
    assert len(keys) < 2 * num_mb * G
