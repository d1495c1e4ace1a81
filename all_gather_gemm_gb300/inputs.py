"""Seeded synthetic inputs for the all-gather matmul workloads.

This module only draws random numbers and casts them to the storage type; it
holds none of the operation's arithmetic, so both the CUDA path's tests and
the CPU oracle can take their inputs from here.

Workloads follow the shapes the pages measure: the cube sweep of the Helion
all-gather-matmul benchmark table (M=N=K from 256 to 4096 in steps of 128,
bf16) and the Iris HBM-buffer result tables (N=3584, K=8192, fp16, M in
{1024, 4096, 16384}, 2/4/8 row shards).

Recipe: one ``torch.Generator`` seeded per workload draws the whole gathered
A ([M, K], fp32) first, then b ([K, N]), then the bias ([N], fp32) when there
is one; A and b are cast to the 16-bit type with torch's round-to-nearest-even
and A is split into D row shards.  The seed is 0 for the small two-shard case
and ``(M*1000003 + N*1009 + K*17 + D) mod 2**31`` for every other shape.

FP8 workloads (an extension, not on the pages) draw the same way, cast A and
b to E4M3 with torch's conversion and keep b transposed ([N, K]), the layout
the FP8 entry takes; their per-tensor scales (``scale_a``, ``scale_b``) are
workload fields, 1/sqrt(K) on b in place of scaling b's values.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
import math

import numpy as np
import torch

_TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16,
                "fp8_e4m3": getattr(torch, "float8_e4m3fn", None)}


@dataclass(frozen=True)
class Workload:
    name: str
    D: int
    m_per_shard: int
    K: int
    N: int
    dtype: str = "bf16"          # storage type of a, b, a_gathered, out
    a_dist: str = "normal"       # "normal" or "uniform"
    a_scale: str = "one"         # "one" or "inv_sqrt_k"
    b_dist: str = "normal"
    b_scale: str = "inv_sqrt_k"
    bias: bool = False
    layouts: tuple = ("k_contiguous",)
    seed: int | None = None      # None: the per-shape rule
    scale_a: float = 1.0         # FP8 only: per-tensor scales passed to the op
    scale_b: float = 1.0

    @property
    def M(self) -> int:
        return self.D * self.m_per_shard

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def resolved_seed(self) -> int:
        if self.seed is not None:
            return self.seed
        return (self.M * 1000003 + self.N * 1009 + self.K * 17 + self.D) % (2 ** 31)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def small_two_shard() -> Workload:
    """Two shards of 128x256, b 256x256, bf16, U[-1,1] for both, seed 0."""
    return Workload("two_shard_256", D=2, m_per_shard=128, K=256, N=256, dtype="bf16",
                    a_dist="uniform", a_scale="one", b_dist="uniform", b_scale="one",
                    seed=0)


def cube(n: int, D: int = 8) -> Workload:
    """M=N=K=n, D row shards, A and b ~ N(0,1)/sqrt(K), bf16."""
    if n % D:
        raise ValueError("n must be a multiple of D")
    return Workload(f"cube_{n}", D=D, m_per_shard=n // D, K=n, N=n, dtype="bf16",
                    a_dist="normal", a_scale="inv_sqrt_k", b_dist="normal",
                    b_scale="inv_sqrt_k")


def cube_sweep() -> list:
    return [cube(n) for n in range(256, 4096 + 1, 128)]


def iris_m1024(D: int) -> Workload:
    """M=1024 N=3584 K=8192 fp16, D shards, A ~ N(0,1), b ~ N(0,1)/sqrt(K)."""
    return Workload(f"m1024_d{D}", D=D, m_per_shard=1024 // D, K=8192, N=3584,
                    dtype="fp16", a_dist="normal", a_scale="one", b_dist="normal",
                    b_scale="inv_sqrt_k")


def iris_m16384() -> Workload:
    """M=16384 N=3584 K=8192 fp16, 8 shards of 2048x8192; both staging layouts."""
    return Workload("m16384_d8", D=8, m_per_shard=2048, K=8192, N=3584, dtype="fp16",
                    a_dist="normal", a_scale="one", b_dist="normal",
                    b_scale="inv_sqrt_k", layouts=("k_contiguous", "m_contiguous"))


def iris_m4096_bias() -> Workload:
    """M=4096 N=3584 K=8192 bf16, 8 shards, A ~ U[-1,1], b ~ U[-1,1]/sqrt(K),
    fp32 bias ~ N(0,1), m-contiguous staging."""
    return Workload("m4096_d8_bias", D=8, m_per_shard=512, K=8192, N=3584, dtype="bf16",
                    a_dist="uniform", a_scale="one", b_dist="uniform",
                    b_scale="inv_sqrt_k", bias=True, layouts=("m_contiguous",))


def iris_m16384_colshard(D: int = 8) -> Workload:
    """Output-sharded form of the M=16384 workload: one rank's column slice,
    N = 3584 / D (b column-sharded), the same gathered A (M=16384, K=8192,
    fp16, D shards).  The gather is unchanged while the GEMM is D times
    smaller."""
    return Workload(f"m16384_d{D}_colshard", D=D, m_per_shard=16384 // D, K=8192,
                    N=3584 // D, dtype="fp16", a_dist="normal", a_scale="one",
                    b_dist="normal", b_scale="inv_sqrt_k")


def fp8_small() -> Workload:
    """FP8 E4M3: two shards of 128x256, b 256x256, U[-1,1], scale_b = 1/16."""
    return Workload("fp8_two_shard_256", D=2, m_per_shard=128, K=256, N=256, dtype="fp8_e4m3",
                    a_dist="uniform", a_scale="one", b_dist="uniform", b_scale="one",
                    seed=1, scale_a=1.0, scale_b=1.0 / 16)


def fp8_m16384() -> Workload:
    """FP8 E4M3 form of the M=16384 N=3584 K=8192 workload (8 shards of 2048 rows):
    A, b ~ N(0,1) in E4M3, scale_b = 1/sqrt(K)."""
    return Workload("fp8_m16384_d8", D=8, m_per_shard=2048, K=8192, N=3584, dtype="fp8_e4m3",
                    a_dist="normal", a_scale="one", b_dist="normal", b_scale="one",
                    scale_b=1.0 / math.sqrt(8192))


def fp8_m1024(D: int = 8) -> Workload:
    """FP8 E4M3, M=1024 N=3584 K=8192, D shards, scale_b = 1/sqrt(K)."""
    return Workload(f"fp8_m1024_d{D}", D=D, m_per_shard=1024 // D, K=8192, N=3584,
                    dtype="fp8_e4m3", a_dist="normal", a_scale="one", b_dist="normal",
                    b_scale="one", scale_b=1.0 / math.sqrt(8192))


def fp8_cube(n: int, D: int = 8) -> Workload:
    """FP8 E4M3, M=N=K=n, D shards, A, b ~ N(0,1), scale_a = scale_b = n^-1/4."""
    return Workload(f"fp8_cube_{n}", D=D, m_per_shard=n // D, K=n, N=n, dtype="fp8_e4m3",
                    a_dist="normal", a_scale="one", b_dist="normal", b_scale="one",
                    scale_a=n ** -0.25, scale_b=n ** -0.25)


def all_workloads() -> list:
    return ([small_two_shard()] + cube_sweep() + [iris_m1024(d) for d in (2, 4, 8)]
            + [iris_m16384(), iris_m4096_bias()])


def _draw(gen: torch.Generator, shape, dist: str) -> torch.Tensor:
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    raise ValueError(dist)


def _scale(t: torch.Tensor, how: str, K: int) -> torch.Tensor:
    if how == "one":
        return t
    if how == "inv_sqrt_k":
        return t * (1.0 / math.sqrt(K))
    raise ValueError(how)


@dataclass
class Inputs:
    workload: Workload
    shards: list          # D torch tensors [m_per_shard, K], 16-bit (or E4M3), CPU, contiguous
    b: torch.Tensor       # [K, N], 16-bit, CPU; E4M3 workloads: [N, K] (transposed)
    bias: torch.Tensor | None  # [N] fp32, CPU

    def bits(self, t: torch.Tensor) -> np.ndarray:
        """A tensor's bit patterns for the oracle: uint16 (16-bit types) or uint8 (E4M3)."""
        if t.element_size() == 1:
            return t.contiguous().view(torch.uint8).numpy()
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    def shard_bits(self) -> list:
        return [self.bits(s) for s in self.shards]

    def b_bits(self) -> np.ndarray:
        return self.bits(self.b)

    def bias_np(self):
        return None if self.bias is None else self.bias.numpy()


def make_inputs(w: Workload) -> Inputs:
    gen = torch.Generator().manual_seed(w.resolved_seed())
    tdt = _TORCH_DTYPE[w.dtype]
    a = _scale(_draw(gen, (w.M, w.K), w.a_dist), w.a_scale, w.K).to(tdt)
    b = _scale(_draw(gen, (w.K, w.N), w.b_dist), w.b_scale, w.K).to(tdt).contiguous()
    if w.dtype == "fp8_e4m3":
        b = b.t().contiguous()  # the FP8 entry takes b as [N, K]
    bias = torch.randn((w.N,), generator=gen, dtype=torch.float32) if w.bias else None
    shards = [a[r * w.m_per_shard:(r + 1) * w.m_per_shard].contiguous() for r in range(w.D)]
    return Inputs(w, shards, b, bias)
