"""Pins of the oracle's FP8 E4M3 extension (CPU): out = bf16(scale_a *
scale_b * (a @ b) + bias) with b given as [N, K].

Independent checks only: the E4M3 decoding against torch's float8_e4m3fn
conversion (a library routine) and against values the format's definition
fixes; the GEMM against exact integer arithmetic, an identity b, a zero A and
the row-block structure of the gathered product.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def test_e4m3_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))  # -0.0 at 0x80


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x40, 2.0), (0x3C, 1.5), (0x30, 0.5),
    (0x7E, 448.0),                 # S.1111.110: the largest finite value
    (0x08, 2.0 ** -6),             # smallest normal
    (0x01, 2.0 ** -9),             # smallest subnormal
    (0x07, 7 * 2.0 ** -9),         # largest subnormal
    (0xB8, -1.0), (0xFE, -448.0),
])
def test_e4m3_values_fixed_by_the_format(code, value):
    assert oracle.e4m3_to_f32(np.array([code], np.uint8))[0] == value


@pytest.mark.parametrize("code", [0x7F, 0xFF])
def test_e4m3_nan_codes(code):
    assert math.isnan(oracle.e4m3_to_f32(np.array([code], np.uint8))[0])


def _e4m3(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_integer_gemm_is_exact():
    """Integers in [-8, 8] are exact in E4M3; with K=512 every partial sum is an
    exact fp32 integer, so the fp32 result equals int64 arithmetic."""
    g = torch.Generator().manual_seed(11)
    M, K, N = 48, 512, 40
    a = torch.randint(-8, 9, (M, K), generator=g)
    b = torch.randint(-8, 9, (K, N), generator=g)
    out32, outb, _, _ = oracle.gemm_rows_fp8(_e4m3(a.float()), _e4m3(b.t().float()))
    exact = (a @ b).numpy()
    assert np.array_equal(out32, exact.astype(np.float32))
    exp_bf16 = torch.from_numpy(exact).float().to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(outb, exp_bf16.view(np.uint16))


def test_scales_multiply_the_sum():
    g = torch.Generator().manual_seed(12)
    M, K, N = 16, 256, 24
    a = torch.randint(-8, 9, (M, K), generator=g)
    b = torch.randint(-8, 9, (K, N), generator=g)
    out32, _, _, _ = oracle.gemm_rows_fp8(_e4m3(a.float()), _e4m3(b.t().float()), 2.0, 0.25)
    assert np.array_equal(out32, (0.5 * (a @ b).numpy()).astype(np.float32))


def test_identity_b_returns_a():
    g = torch.Generator().manual_seed(13)
    K = 64
    a8 = _e4m3(torch.randn(32, K, generator=g))
    eye = _e4m3(torch.eye(K))
    out32, _, _, _ = oracle.gemm_rows_fp8(a8, eye)
    assert np.array_equal(out32, oracle.e4m3_to_f32(a8))


def test_zero_a_gives_the_bias():
    N, K = 24, 32
    bias = np.linspace(-3, 3, N).astype(np.float32)
    bt = _e4m3(torch.randn(N, K, generator=torch.Generator().manual_seed(14)))
    out32, outb, _, _ = oracle.gemm_rows_fp8(np.zeros((8, K), np.uint8), bt, 1.0, 1.0, bias)
    assert np.array_equal(out32, np.broadcast_to(bias, (8, N)))


def test_row_blocks_equal_the_shard_products():
    g = torch.Generator().manual_seed(15)
    D, m, K, N = 3, 20, 96, 40
    shards = [_e4m3(torch.randn(m, K, generator=g)) for _ in range(D)]
    bt = _e4m3(torch.randn(N, K, generator=g))
    a = oracle.all_gather_bytes(shards)
    assert np.array_equal(a, np.concatenate(shards))
    full, _, _, _ = oracle.gemm_rows_fp8(a, bt, 0.5, 2.0)
    for r in range(D):
        part, _, _, _ = oracle.gemm_rows_fp8(shards[r], bt, 0.5, 2.0)
        assert np.array_equal(full[r * m:(r + 1) * m], part)


def test_abs_term_carries_the_scale():
    a = _e4m3(torch.tensor([[1.0, -2.0]]))
    bt = _e4m3(torch.tensor([[3.0, 4.0]]))
    out32, _, abs_ab, _ = oracle.gemm_rows_fp8(a, bt, -0.5, 1.0)
    assert out32[0, 0] == -0.5 * (3.0 - 8.0)
    assert abs_ab[0, 0] == 0.5 * (3.0 + 8.0)
