"""Pins for the CPU oracle (no GPU).

The oracle restates the op's plain definition -- a = row concatenation of the
shards, out = a @ b (+ bias) with fp32 accumulation and one RNE rounding --
and these tests tie it to things other than itself: torch's own 16-bit casts,
numpy's concatenate and float64 matmul, exact integer arithmetic, hand-worked
examples, and identities (identity / permutation / one-hot b, zero b with a
bias, per-shard row blocks).  Each is chosen so that a plausible slip in the
oracle -- a dropped k term, a transposed or mis-indexed operand, a wrong shard
order, a bias on the wrong column, a rounding that is not to-nearest-even --
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
TDT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 values -> 16-bit patterns via torch's cast (an independent RNE)."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(TDT[dtype])
    return t.view(torch.int16).numpy().view(np.uint16)


def widen(bits: np.ndarray, dtype: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TDT[dtype])
    return t.float().numpy()


def split(a_bits, D):
    m = a_bits.shape[0] // D
    return [np.ascontiguousarray(a_bits[r * m:(r + 1) * m]) for r in range(D)]


# ---------------------------------------------------------------- conversions

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_widen_every_pattern_matches_torch(oracle_mod, dtype):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.to_f32(bits, dtype)
    ref = widen(bits, dtype)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_round_matches_torch(oracle_mod, dtype):
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 1 << 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    vals = [raw.view(np.float32)]
    # values spread over the 16-bit type's range, incl. subnormals and overflow
    vals.append((rng.standard_normal(200_000) * 10.0 ** rng.uniform(-9, 6, 200_000))
                .astype(np.float32))
    # exact ties: every 16-bit value plus half of its quantum
    all16 = widen(np.arange(1 << 16, dtype=np.uint32).astype(np.uint16), dtype)
    fin = all16[np.isfinite(all16)].astype(np.float64)
    nxt = np.nextafter(fin.astype(np.float32), np.float32(np.inf)).astype(np.float64)
    vals.append(fin.astype(np.float32))
    step = (widen(to_bits(fin.astype(np.float32), dtype) + 1, dtype).astype(np.float64) - fin)
    ties = (fin + step / 2).astype(np.float32)
    vals.append(ties[np.isfinite(ties)])
    vals.append(nxt.astype(np.float32))
    vals.append(np.array([0.0, -0.0, np.inf, -np.inf, 65504, 65519.99, 65520, 65536,
                          6e-8, 5.96e-8, 2.98e-8, 2.99e-8, 3.4e38, 1e-45], np.float32))
    x = np.concatenate(vals)
    x = x[~np.isnan(x)]
    ours = oracle_mod.from_f32(x, dtype)
    ref = to_bits(x, dtype)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, (x[bad[:5]], ours[bad[:5]], ref[bad[:5]])
    assert np.isnan(oracle_mod.to_f32(oracle_mod.from_f32(np.array([np.nan], np.float32),
                                                          dtype), dtype)).all()


# ---------------------------------------------------------------- gather

@pytest.mark.parametrize("D,m,K", [(1, 3, 8), (2, 128, 256), (3, 5, 16), (8, 32, 24)])
def test_all_gather_is_numpy_concatenate(oracle_mod, D, m, K):
    rng = np.random.default_rng(D * 100 + m)
    shards = [rng.integers(0, 1 << 16, size=(m, K), dtype=np.uint32).astype(np.uint16)
              for _ in range(D)]
    got = oracle_mod.all_gather(shards)
    assert np.array_equal(got, np.concatenate(shards, axis=0))


# ---------------------------------------------------------------- hand-worked

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_worked_examples(oracle_mod, case):
    dt = case["dtype"]
    shards = [to_bits(np.array(s, np.float32), dt) for s in case["shards"]]
    b = to_bits(np.array(case["b"], np.float32), dt)
    bias = None if case["bias"] is None else np.array(case["bias"], np.float32)
    a, out_f32, out, _ = oracle_mod.ag_matmul(shards, b, bias, dtype=dt)
    assert np.array_equal(a, to_bits(np.array(case["a_gathered"], np.float32), dt))
    assert np.array_equal(out_f32, np.array(case["out_f32"], np.float32))
    want = np.array([int(v, 16) for v in case["out_bits"]], np.uint16).reshape(out.shape)
    assert np.array_equal(out, want)


# ---------------------------------------------------------------- exact integer brute force

def _int_case(rng, D, m, K, N, lo, hi, dtype, with_bias):
    a = rng.integers(lo, hi + 1, size=(D * m, K)).astype(np.float32)
    b = rng.integers(lo, hi + 1, size=(K, N)).astype(np.float32)
    bias = rng.integers(-8, 9, size=(N,)).astype(np.float32) if with_bias else None
    return a, b, bias


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D,m,K,N,bias", [(1, 4, 4, 4, False), (2, 2, 4, 4, False),
                                          (4, 1, 4, 4, True), (3, 5, 7, 9, True),
                                          (2, 3, 64, 5, False)])
def test_integer_brute_force_exact(oracle_mod, dtype, D, m, K, N, bias):
    """Integer entries in [-4, 4]: every product and partial sum is a small
    integer, exact in fp32, so the oracle must equal integer arithmetic."""
    rng = np.random.default_rng(K * 31 + N)
    a, b, bvec = _int_case(rng, D, m, K, N, -4, 4, dtype, bias)
    shards = split(to_bits(a, dtype), D)
    _, out_f32, out, abs_ab = oracle_mod.ag_matmul(shards, to_bits(b, dtype), bvec, dtype=dtype)
    ai, bi = a.astype(np.int64).tolist(), b.astype(np.int64).tolist()
    exact = [[sum(ai[i][k] * bi[k][j] for k in range(K)) + (int(bvec[j]) if bias else 0)
              for j in range(N)] for i in range(D * m)]
    exact_abs = [[sum(abs(ai[i][k]) * abs(bi[k][j]) for k in range(K)) for j in range(N)]
                 for i in range(D * m)]
    assert np.array_equal(out_f32, np.array(exact, np.float32))
    assert np.array_equal(abs_ab, np.array(exact_abs, np.float32))
    assert np.array_equal(out, to_bits(np.array(exact, np.float32), dtype))


# ---------------------------------------------------------------- D = 1 is a plain GEMM

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_single_shard_is_plain_gemm_within_fp32_bound(oracle_mod, dtype):
    rng = np.random.default_rng(7)
    M, K, N = 48, 640, 72
    a = to_bits(rng.standard_normal((M, K)).astype(np.float32), dtype)
    b = to_bits((rng.standard_normal((K, N)) / math.sqrt(K)).astype(np.float32), dtype)
    _, out_f32, out, abs_ab = oracle_mod.ag_matmul([a], b, dtype=dtype)
    a64, b64 = widen(a, dtype).astype(np.float64), widen(b, dtype).astype(np.float64)
    ref = a64 @ b64
    # recursive fp32 summation: |err| <= K * 2^-24 * sum|a||b| (+ tiny slack)
    bound = K * 2.0 ** -24 * (np.abs(a64) @ np.abs(b64)) * 1.01
    assert np.all(np.abs(out_f32 - ref) <= bound)
    assert np.allclose(abs_ab, np.abs(a64) @ np.abs(b64), rtol=1e-5)
    # the stored result is the RNE of the fp32 sum
    assert np.array_equal(out, to_bits(out_f32, dtype))


# ---------------------------------------------------------------- row blocks = per-shard GEMMs

@pytest.mark.parametrize("D", [2, 3, 8])
def test_row_block_r_is_shard_r_times_b(oracle_mod, D):
    rng = np.random.default_rng(D)
    m, K, N = 16, 96, 40
    shards = [to_bits(rng.uniform(-1, 1, (m, K)).astype(np.float32), "bf16")
              for _ in range(D)]
    b = to_bits(rng.uniform(-1, 1, (K, N)).astype(np.float32), "bf16")
    bias = rng.standard_normal(N).astype(np.float32)
    _, full32, full, _ = oracle_mod.ag_matmul(shards, b, bias, dtype="bf16")
    for r in range(D):
        _, p32, p, _ = oracle_mod.ag_matmul([shards[r]], b, bias, dtype="bf16")
        assert np.array_equal(full32[r * m:(r + 1) * m], p32)
        assert np.array_equal(full[r * m:(r + 1) * m], p)


def test_sampled_rows_equal_full_rows(oracle_mod):
    rng = np.random.default_rng(3)
    shards = [to_bits(rng.standard_normal((8, 64)).astype(np.float32), "fp16")
              for _ in range(4)]
    b = to_bits(rng.standard_normal((64, 24)).astype(np.float32), "fp16")
    _, f32, f, _ = oracle_mod.ag_matmul(shards, b, dtype="fp16")
    rows = np.array([31, 0, 17, 8, 8], np.int64)
    _, s32, s, _ = oracle_mod.ag_matmul(shards, b, dtype="fp16", rows=rows)
    assert np.array_equal(s32, f32[rows]) and np.array_equal(s, f[rows])


# ---------------------------------------------------------------- identity, permutation, one-hot

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_identity_b_returns_gathered_a(oracle_mod, dtype):
    rng = np.random.default_rng(11)
    K = 40
    shards = [to_bits(rng.standard_normal((6, K)).astype(np.float32), dtype) for _ in range(3)]
    b = to_bits(np.eye(K, dtype=np.float32), dtype)
    a, _, out, _ = oracle_mod.ag_matmul(shards, b, dtype=dtype)
    assert np.array_equal(out, a)


def test_permutation_b_permutes_columns(oracle_mod):
    """b[k, p[k]] = 1: out[:, p[k]] = a[:, k].  A transposed b would apply the
    inverse permutation instead, which differs for this p."""
    rng = np.random.default_rng(12)
    K = 24
    p = rng.permutation(K)
    assert not np.array_equal(p, np.argsort(p))
    P = np.zeros((K, K), np.float32)
    P[np.arange(K), p] = 1.0
    shards = [to_bits(rng.standard_normal((5, K)).astype(np.float32), "bf16") for _ in range(2)]
    a, _, out, _ = oracle_mod.ag_matmul(shards, to_bits(P, "bf16"), dtype="bf16")
    assert np.array_equal(out[:, p], a)


def test_one_hot_row_of_b_selects_a_column(oracle_mod):
    rng = np.random.default_rng(13)
    K, N, k0 = 32, 20, 9
    B = np.zeros((K, N), np.float32)
    B[k0, :] = 1.0
    shards = [to_bits(rng.standard_normal((7, K)).astype(np.float32), "fp16") for _ in range(2)]
    a, _, out, _ = oracle_mod.ag_matmul(shards, to_bits(B, "fp16"), dtype="fp16")
    assert np.array_equal(out, np.repeat(a[:, k0:k0 + 1], N, axis=1))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_zero_b_gives_rounded_bias(oracle_mod, dtype):
    rng = np.random.default_rng(14)
    N = 33
    bias = rng.standard_normal(N).astype(np.float32)
    shards = [to_bits(rng.standard_normal((3, 16)).astype(np.float32), dtype) for _ in range(2)]
    b = np.zeros((16, N), np.uint16)
    _, f32, out, _ = oracle_mod.ag_matmul(shards, b, bias, dtype=dtype)
    assert np.array_equal(f32, np.tile(bias, (6, 1)))
    assert np.array_equal(out, np.tile(to_bits(bias, dtype), (6, 1)))


# ---------------------------------------------------------------- tolerance helper

def test_within_tolerance_flags_first_violation(oracle_mod):
    ref = np.zeros((3, 4), np.float32)
    scale = np.ones((3, 4), np.float32)
    got = ref.copy()
    ok, ratio, idx = oracle_mod.within_tolerance(got, ref, scale)
    assert ok and ratio == 0 and idx is None
    got[1, 2] = 0.02
    ok, ratio, idx = oracle_mod.within_tolerance(got, ref, scale)
    assert not ok and idx == (1, 2) and ratio > 1
    got[1, 2] = np.nan
    assert not oracle_mod.within_tolerance(got, ref, scale)[0]
