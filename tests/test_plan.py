"""The launch plan of fused calls (ag_plan_fused), on the CPU: the fetch
prologue, the L2 prefetch of small A, CTA pairs and k_per_flag are chosen as
the library documents, for a GB300 (152 SMs, 76 co-resident CTA pairs)."""
import pytest

import all_gather_gemm_gb300 as agmm

SMS, PAIRS = 152, 76


def plan(D, m, K, N, **kw):
    return agmm.plan_fused(D, m, K, N, SMS, PAIRS, **kw)


def test_headline_shape_runs_neither_prologue_nor_prefetch():
    p = plan(8, 2048, 8192, 3584, dtype="fp16")
    assert p == {"grid": 152, "cta_pairs": 1, "tiles": 64 * 14, "k_per_flag": 8,
                 "prologue_cta0": -1, "l2_prefetch": 0, "block_m": 256, "stages": 6,
                 "k_ascending": 1}


@pytest.mark.parametrize("n", [2176, 2304, 2432, 2560, 2688, 2816, 3200, 3328])
def test_cube_shapes_with_a_partial_last_wave_run_the_prologue(n):
    # pair tiles T on 76 pairs: the last 76 - T % 76 pairs have one tile fewer
    p = plan(8, n // 8, n, n)
    T = -(-(-(-n // 128)) // 2) * -(-n // 256)
    assert p["tiles"] == T and p["grid"] == 152
    assert 76 < T <= 3 * 76 and T % 76
    assert p["prologue_cta0"] == 2 * (T % 76)
    assert p["l2_prefetch"] == (n * n * 2 <= 12 << 20)


@pytest.mark.parametrize("n", [2944, 3072, 3456, 3584, 4096])
def test_cube_shapes_without_prologue(n):
    # 2944 / 3072: too few spare CTAs for A; 3456 ...: A too large per spare CTA
    # or more than three waves
    assert plan(8, n // 8, n, n)["prologue_cta0"] == -1


@pytest.mark.parametrize("n", [256, 1024, 2048])
def test_one_wave_cubes(n):
    """K of at most 32 k-blocks and every 128-row tile in one wave: single
    CTAs (128 x 256 tiles), one per tile."""
    p = plan(8, n // 8, n, n)
    T = (n // 128) * (n // 256)
    assert (p["cta_pairs"], p["block_m"], p["stages"]) == (0, 128, 4)
    assert p["tiles"] == T and p["grid"] == T and p["prologue_cta0"] == -1
    assert p["l2_prefetch"] == 1
    num_kb, num_nb = n // 64, n // 256
    assert p["k_per_flag"] == min(num_kb, min(8, max(4, num_kb // num_nb)))
    # the tile options still force CTA pairs
    q = plan(8, n // 8, n, n, block_m=256)
    assert q["cta_pairs"] == 1 and q["tiles"] == (n // 256) * (n // 256) and q["grid"] == 2 * q["tiles"]


@pytest.mark.parametrize("D,m,K,N,single", [
    (8, 256, 2048, 2048, True),     # cube 2048: 32 k-blocks, 128 tiles
    (8, 272, 2176, 2176, False),    # cube 2176: 34 k-blocks
    (8, 128, 8192, 3584, False),    # M=1024 K=8192: one wave, long K
    (8, 2048, 2048, 3584, False),   # K short but 128 x 14 tiles: more than one wave
    (2, 128, 256, 256, True),       # the two-shard case
])
def test_automatic_tile_shape(D, m, K, N, single):
    p = plan(D, m, K, N)
    assert p["cta_pairs"] == (0 if single else 1)
    assert p["block_m"] == (128 if single else 256)
    # FP8 counts K in bytes: the same rule on K/2 16-bit words
    if K % 16 == 0:
        assert plan(D, m, 2 * K, N, dtype="fp8_e4m3")["cta_pairs"] == (0 if single else 1)


def test_m_contiguous_and_fp8():
    assert plan(8, 304, 2432, 2432, layout="m_contiguous")["prologue_cta0"] == -1
    p = plan(8, 2048, 8192, 3584, dtype="fp8_e4m3")
    assert p["tiles"] == 64 * 14 and p["k_per_flag"] == 8 and p["prologue_cta0"] == -1
    # FP8 A of 8 MB (bytes) is prefetched
    assert plan(8, 128, 8192, 3584, dtype="fp8_e4m3")["l2_prefetch"] == 1


def test_restricted_grids():
    p = plan(4, 384, 520, 1024, num_sms=40)  # 24 pair tiles on 20 pairs
    assert p["grid"] == 40 and p["tiles"] == 24 and p["prologue_cta0"] == 8
    p = plan(4, 160, 1024, 512, num_sms=1)
    assert p["cta_pairs"] == 0 and p["grid"] == 1 and p["tiles"] == 10
    assert agmm.plan_fused(4, 160, 1024, 512, SMS, 0)["cta_pairs"] == 0


@pytest.mark.parametrize("D,m,K,N,waves4", [(8, 2048, 8192, 3584, True), (8, 512, 8192, 3584, False),
                                            (8, 512, 4096, 4096, False), (8, 128, 8192, 3584, False),
                                            (8, 1024, 8192, 7168, True)])
def test_k_order_by_wave_count(D, m, K, N, waves4):
    """Calls of four or more waves run every tile k ascending, in both
    layouts; fewer waves keep each tile's owned k-range first (the fetch
    prologue, which owns nothing, runs k ascending without this flag)."""
    p = plan(D, m, K, N, dtype="fp16")
    assert (p["tiles"] >= 4 * p["grid"] // 2) == waves4
    assert p["k_ascending"] == int(waves4)
    assert plan(D, m, K, N, layout="m_contiguous")["k_ascending"] == int(waves4)


def test_tile_options_choose_the_compiled_variant():
    """block_m 128 (or stages 4) selects single CTAs with 128 x 256 tiles,
    block_m 256 (or stages 6) CTA pairs; 256-row tiles need a CTA pair."""
    for kw in ({"block_m": 128}, {"stages": 4}, {"block_m": 128, "stages": 4}):
        p = plan(8, 2048, 8192, 3584, dtype="fp16", **kw)
        assert (p["cta_pairs"], p["block_m"], p["stages"], p["grid"]) == (0, 128, 4, 152), kw
        assert p["tiles"] == 128 * 14
    for kw in ({"block_m": 256}, {"stages": 6}, {"block_n": 256, "block_k": 64,
                                                 "producer_warps": 4}):
        p = plan(8, 2048, 8192, 3584, dtype="fp16", **kw)
        assert (p["cta_pairs"], p["block_m"], p["stages"]) == (1, 256, 6), kw
    with pytest.raises(agmm.AgmmError) as e:
        plan(4, 160, 1024, 512, num_sms=1, block_m=256)
    assert e.value.status == 2
    with pytest.raises(agmm.AgmmError) as e:
        agmm.plan_fused(4, 160, 1024, 512, SMS, 0, stages=6)
    assert e.value.status == 2
    for kw in ({"block_m": 192}, {"stages": 3}, {"block_n": 128}, {"producer_warps": 2},
               {"block_m": 128, "stages": 6}):
        with pytest.raises(agmm.AgmmError) as e:
            plan(8, 2048, 8192, 3584, **kw)
        assert e.value.status == 2, kw
    assert plan(8, 2048, 16384, 3584, dtype="fp8_e4m3", block_k=128)["block_m"] == 256


def test_rejections():
    with pytest.raises(agmm.AgmmError):
        plan(0, 128, 256, 256)
    with pytest.raises(agmm.AgmmError):
        plan(2, 128, 260, 256)  # K % 8
    with pytest.raises(agmm.AgmmError):
        plan(17, 128, 256, 256)  # more than AG_MAX_SHARDS
    with pytest.raises(agmm.AgmmError):
        agmm.plan_fused(2, 128, 256, 256, 0, 76)
