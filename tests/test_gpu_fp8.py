"""GPU parity of the FP8 E4M3 extension (through the C ABI) against the CPU oracle.

out = bf16(scale_a * scale_b * (a @ b) + bias) with b given as [N, K].
a_gathered must be byte-exact; out must satisfy, elementwise,
    |out - ref_f32| <= 1e-2 * |s| (|a|.|b|)_ij + 1e-3 + 2^-8 |ref_f32|
(the 16-bit bound with the scale s = scale_a*scale_b carried into the |a|.|b|
term, plus the bf16 output's rounding, at most half an ulp = 2^-9 relative,
doubled).  Fused and barrier paths are both checked; the fused kernel's
results are bitwise equal across local ranks.
"""
import numpy as np
import pytest
import torch

import all_gather_gemm_gb300 as agmm
from all_gather_gemm_gb300 import inputs as inp

pytestmark = pytest.mark.gpu

REL, ATOL, ROUND = 1e-2, 1e-3, 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    agmm.library()
    yield


def u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.uint8).numpy()


def run(x: inp.Inputs, fused=True, rank=0, **kw):
    w = x.workload
    shards = [s.cuda() for s in x.shards]
    bias = x.bias.cuda() if x.bias is not None else None
    fn = agmm.ag_matmul if fused else agmm.ag_then_matmul
    extra = {"rank": rank} if fused else {}
    a_g, out = fn(shards, x.b.cuda(), bias, scale_a=w.scale_a, scale_b=w.scale_b, **extra, **kw)
    code, info = agmm.device_error()
    assert code == 0, f"device error {code} info {info:#x}"
    return a_g, out


def check(oracle, x: inp.Inputs, results, rows=None):
    w = x.workload
    exp_a = oracle.all_gather_bytes(x.shard_bits())
    ref32, _, absab, _ = oracle.gemm_rows_fp8(exp_a, x.b_bits(), w.scale_a, w.scale_b,
                                              x.bias_np(), rows=rows)
    bound = REL * absab.astype(np.float64) + ATOL + ROUND * np.abs(ref32.astype(np.float64))
    for a_d, o_d, label in results:
        assert o_d.dtype == torch.bfloat16
        got_a = u8(a_d)
        assert np.array_equal(got_a, exp_a), f"{label}: a_gathered differs"
        got = o_d if rows is None else o_d[torch.as_tensor(rows, device=o_d.device)]
        err = np.abs(got.float().cpu().numpy().astype(np.float64) - ref32)
        bad = ~(err <= bound)
        assert not bad.any(), (f"{label}: out outside tolerance at {np.argwhere(bad)[:3]} "
                               f"(worst err/bound {np.nanmax(err / bound):.3g})")


def test_fp8_small(oracle_mod):
    x = inp.make_inputs(inp.fp8_small())
    check(oracle_mod, x, [(*run(x), "fused"), (*run(x, fused=False), "barrier")])


RAGGED = [
    # (D, m_per_shard, K, N, bias): several tiles, ragged row blocks and a partial
    # last k-block; m=16 straddles 128-row blocks with 16-row boxes, m=100 takes
    # the register fetcher (shard boundaries off the 8-row grid); K=16 is the minimum.
    (3, 200, 512, 384, True),
    (1, 64, 16, 8, False),
    (5, 130, 1040, 520, True),
    (8, 16, 256, 264, False),
    (7, 100, 3008, 40, True),
    (16, 40, 128, 72, False),  # the maximum shard count
]


@pytest.mark.parametrize("D,m,K,N,bias", RAGGED)
def test_fp8_ragged(oracle_mod, D, m, K, N, bias):
    w = inp.Workload(f"fp8_ragged_{D}_{m}_{K}_{N}", D=D, m_per_shard=m, K=K, N=N,
                     dtype="fp8_e4m3", a_dist="uniform", b_dist="uniform", b_scale="one",
                     bias=bias, scale_a=0.75, scale_b=0.5)
    x = inp.make_inputs(w)
    res = []
    first = None
    for rank in sorted({0, D - 1}):
        a_f, o_f = run(x, rank=rank)
        res.append((a_f, o_f, f"fused rank {rank}"))
        if first is None:
            first = o_f
        else:
            assert torch.equal(o_f, first), "fused output depends on the local rank"
    res.append((*run(x, fused=False), "barrier"))
    check(oracle_mod, x, res)


@pytest.mark.parametrize("num_sms", [1, 3])
def test_fp8_small_grids(oracle_mod, num_sms):
    """Grids below two SMs run the single-CTA kernels (b boxes of 256 rows)."""
    w = inp.Workload("fp8_grid", D=3, m_per_shard=160, K=384, N=520, dtype="fp8_e4m3",
                     a_dist="normal", b_dist="normal", b_scale="one", bias=True,
                     scale_b=0.05)
    x = inp.make_inputs(w)
    check(oracle_mod, x, [(*run(x, num_sms=num_sms), "fused"),
                          (*run(x, fused=False, num_sms=num_sms), "barrier")])


def test_fp8_fetch_prologue(oracle_mod):
    """On 40 SMs this call takes two waves, the second partial: the CTAs with
    one tile fewer stage all of A first (the fetch prologue).  k then runs in
    ascending order, as in the barrier GEMM, so the two agree bitwise."""
    w = inp.Workload("fp8_prologue", D=4, m_per_shard=384, K=1040, N=1024, dtype="fp8_e4m3",
                     a_dist="uniform", b_dist="uniform", b_scale="one", bias=True,
                     scale_a=0.75, scale_b=0.5)
    x = inp.make_inputs(w)
    a_f, o_f = run(x, rank=2, num_sms=40)
    a_b, o_b = run(x, fused=False)
    assert torch.equal(o_f, o_b), "fused (prologue) and barrier differ"
    check(oracle_mod, x, [(a_f, o_f, "fused, fetch prologue"), (a_b, o_b, "barrier")])


def test_fp8_integer_inputs_exact():
    """Integers in [-8, 8] and K=512: the fp32 sums are exact, so out must be
    the bf16 rounding of the exact integer result (scaled by 2 * 0.25)."""
    g = torch.Generator().manual_seed(21)
    D, m, K, N = 2, 192, 512, 264
    a = torch.randint(-8, 9, (D * m, K), generator=g)
    b = torch.randint(-8, 9, (K, N), generator=g)
    a8 = a.float().to(torch.float8_e4m3fn)
    bt8 = b.t().contiguous().float().to(torch.float8_e4m3fn)
    shards = [a8[r * m:(r + 1) * m].contiguous().cuda() for r in range(D)]
    exact = (0.5 * (a @ b).double()).float().to(torch.bfloat16)
    for fn in (agmm.ag_matmul, agmm.ag_then_matmul):
        _, out = fn(shards, bt8.cuda(), scale_a=2.0, scale_b=0.25)
        assert agmm.device_error() == (0, 0)
        assert torch.equal(out.cpu(), exact)


def test_fp8_identity_b_returns_gathered_a():
    g = torch.Generator().manual_seed(22)
    D, m, K = 4, 96, 256
    shards = [torch.randn(m, K, generator=g).to(torch.float8_e4m3fn).cuda() for _ in range(D)]
    eye = torch.eye(K).to(torch.float8_e4m3fn).cuda()
    a_g, out = agmm.ag_matmul(shards, eye, rank=1)
    assert agmm.device_error() == (0, 0)
    assert np.array_equal(u8(a_g), u8(torch.cat(shards)))
    assert torch.equal(out.cpu(), torch.cat(shards).cpu().float().to(torch.bfloat16))


@pytest.mark.parametrize("make", [lambda: inp.fp8_m1024(8), inp.fp8_m16384],
                         ids=["fp8_m1024_d8", "fp8_m16384_d8"])
def test_fp8_iris_shapes_full(oracle_mod, make):
    """Every output element of the Iris shapes in FP8, fused and barrier."""
    w = make()
    x = inp.make_inputs(w)
    check(oracle_mod, x, [(*run(x), "fused"), (*run(x, fused=False), "barrier")])


def test_fp8_rejections():
    g = torch.Generator().manual_seed(23)
    shards = [torch.randn(64, 64, generator=g).to(torch.float8_e4m3fn).cuda() for _ in range(2)]
    bt = torch.randn(64, 64, generator=g).to(torch.float8_e4m3fn).cuda()
    with pytest.raises(agmm.AgmmError) as e:
        agmm.ag_matmul(shards, bt, layout="m_contiguous")
    assert e.value.status == 2  # unsupported
    with pytest.raises(agmm.AgmmError) as e:
        agmm.ag_matmul(shards, bt, scale_a=float("inf"))
    assert e.value.status == 1  # invalid
    odd = [torch.randn(64, 24, generator=g).to(torch.float8_e4m3fn).cuda() for _ in range(2)]
    with pytest.raises(agmm.AgmmError) as e:
        agmm.ag_matmul(odd, torch.randn(64, 24, generator=g).to(torch.float8_e4m3fn).cuda())
    assert e.value.status == 1  # K % 16 != 0
    assert agmm.device_error() == (0, 0)


@pytest.mark.parametrize("chunks", [1, 3])
def test_fp8_chunked_pipeline_equals_barrier(oracle_mod, chunks):
    """The chunked pipeline runs the barrier's GEMM core (k ascending) per chunk,
    so its FP8 result is bitwise the barrier's."""
    w = inp.Workload("fp8_chunked", D=3, m_per_shard=384, K=512, N=264, dtype="fp8_e4m3",
                     a_dist="normal", b_dist="normal", b_scale="one", bias=True, scale_b=0.04)
    x = inp.make_inputs(w)
    shards = [s.cuda() for s in x.shards]
    bias = x.bias.cuda()
    a_c, o_c = agmm.ag_chunked_matmul(shards, x.b.cuda(), bias, chunks=chunks,
                                      scale_a=w.scale_a, scale_b=w.scale_b)
    assert agmm.device_error() == (0, 0)
    a_b, o_b = run(x, fused=False)
    assert torch.equal(o_c, o_b)
    check(oracle_mod, x, [(a_c, o_c, f"chunked {chunks}")])
