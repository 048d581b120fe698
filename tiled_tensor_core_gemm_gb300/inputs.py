"""Seeded synthetic operands for the GEMM workloads.

This module only draws random numbers and lays them out; it holds none of the
GEMM's arithmetic, so both the CUDA path and the oracle can be fed from it.

Recipe (the workloads are synthetic square and ragged GEMMs, as in the
"Learn CuTeDSL" TFLOPS table and the ch. 13 traffic table):

* one CPU ``torch.Generator`` seeded with the workload's seed; A (M x K) is
  drawn first, then B (K x N), from the same generator;
* ``uniform`` is U[-1, 1) = 2*rand - 1, ``normal`` is N(0, 1) via randn;
* for BF16 (FP16, FP8 E4M3 / E5M2) operands the FP32 draw is rounded once to
  that format by round to nearest even, the library's own ``.to(...)``; those
  values are the ground truth for every check;
* ``ints`` draws integers uniformly from [-lo_hi, lo_hi], for the exactness
  tests (every product and partial sum is then an exact small integer).

For the fused epilogue, ``make_epilogue_inputs`` draws the old C (N(0,1),
rounded once to the output type) and the bias (N(0,1) FP32) from a generator
of their own, seeded separately from A and B.

Every array is row-major; ``ld_pad`` adds unused trailing columns so the
leading dimension exceeds the logical width (the padding is filled with NaN so
any read of it shows up in the result).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: str          # "fp32" | "tf32" | "bf16" | "fp16" | "e4m3" | "e5m2"  (the arithmetic path)
    dist: str           # "uniform" | "normal"
    seed: int


# The five published workloads (shapes, distributions and seeds as stated there).
C1_FP32_256 = Workload("fp32 256^3 U[-1,1] seed 0", 256, 256, 256, "fp32", "uniform", 0)
C2_FP32_1024 = Workload("fp32 1024^3 U[-1,1] seed 1", 1024, 1024, 1024, "fp32", "uniform", 1)
C2_TF32_1024 = Workload("tf32 1024^3 U[-1,1] seed 1", 1024, 1024, 1024, "tf32", "uniform", 1)
C3_FP32_4096 = Workload("fp32 4096^3 N(0,1) seed 2", 4096, 4096, 4096, "fp32", "normal", 2)
C3_TF32_4096 = Workload("tf32 4096^3 N(0,1) seed 2", 4096, 4096, 4096, "tf32", "normal", 2)
C4_BF16_8192 = Workload("bf16 8192^3 N(0,1) seed 3", 8192, 8192, 8192, "bf16", "normal", 3)
# FP16 inputs at the pages' own benchmark sizes (their TFLOPS table is FP16 at
# 4096^3, their Nsight comparison FP16 at 8192^3), N(0,1) rounded to FP16.
FP16_4096 = Workload("fp16 4096^3 N(0,1) seed 5", 4096, 4096, 4096, "fp16", "normal", 5)
FP16_8192 = Workload("fp16 8192^3 N(0,1) seed 6", 8192, 8192, 8192, "fp16", "normal", 6)
# FP8 inputs (OCP E4M3 and E5M2) at the same two sizes, N(0,1) rounded to FP8.
E4M3_4096 = Workload("e4m3 4096^3 N(0,1) seed 7", 4096, 4096, 4096, "e4m3", "normal", 7)
E4M3_8192 = Workload("e4m3 8192^3 N(0,1) seed 8", 8192, 8192, 8192, "e4m3", "normal", 8)
E5M2_8192 = Workload("e5m2 8192^3 N(0,1) seed 9", 8192, 8192, 8192, "e5m2", "normal", 9)
C5_BF16_RAGGED = tuple(
    Workload(f"bf16 {m}x{n}x{k} U[-1,1] seed 4", m, n, k, "bf16", "uniform", 4)
    for (m, n, k) in ((1000, 1000, 1000), (4097, 4095, 4099), (16384, 1024, 4096), (128, 8192, 8192))
)


@dataclass(frozen=True)
class GroupedWorkload:
    """A batch of independent GEMMs C_g = A_g . B_g (M_g x K_g times K_g x N);
    K_g = K unless Ks gives one per group."""
    name: str
    Ms: tuple
    N: int
    K: int
    dtype: str
    dist: str
    seed: int
    Ks: tuple = ()

    def k_of(self, g: int) -> int:
        return self.Ks[g] if self.Ks else self.K

    @property
    def flops(self) -> float:
        return 2.0 * sum(m * self.k_of(g) for g, m in enumerate(self.Ms)) * self.N


def skewed_group_rows(total: int, groups: int, seed: int, sigma: float = 0.75) -> tuple:
    """Row counts of `groups` GEMMs summing to `total`: shares proportional to
    seeded lognormal(0, sigma) weights (the uneven token counts a batch of
    experts sees), floored, the remainder added to the largest."""
    rng = np.random.default_rng(seed)
    w = rng.lognormal(0.0, sigma, groups)
    Ms = np.floor(total * w / w.sum()).astype(np.int64)
    Ms[int(np.argmax(Ms))] += total - int(Ms.sum())
    return tuple(int(m) for m in Ms)


# 16 GEMMs of skewed row counts (32768 rows in all) against their own
# 4096 x 4096 B: the same 1.1 TFLOP as the 8192^3 GEMM, as one grouped launch.
GROUPED_BF16 = GroupedWorkload("grouped bf16 16 groups, sum M = 32768, N = K = 4096, lognormal(0, 0.75) row "
                               "shares, N(0,1), seed 10", skewed_group_rows(32768, 16, 10), 4096, 4096, "bf16",
                               "normal", 10)


def skewed_group_depths(groups: int, seed: int, lo: int = 512, hi: int = 8192) -> tuple:
    """K of each group: log-uniform between lo and hi, rounded to a multiple of 64."""
    rng = np.random.default_rng(seed)
    ks = np.exp(rng.uniform(np.log(lo), np.log(hi), groups))
    return tuple(int(max(64, round(k / 64) * 64)) for k in ks)


# The same 16 GEMMs with K differing per group (log-uniform in [512, 8192]):
# work units of unequal cost, where a dynamic schedule can balance the load.
GROUPED_BF16_SKEWK = GroupedWorkload("grouped bf16 16 groups, M = 2048, N = 4096, K log-uniform in [512, 8192], "
                                     "N(0,1), seed 11", (2048,) * 16, 4096, 0, "bf16", "normal", 11,
                                     skewed_group_depths(16, 11))


def grouped_operands(w: GroupedWorkload):
    """[(A_g, B_g)]: group g drawn by make_operands with seed w.seed + g."""
    return [make_operands(m, w.N, w.k_of(g), w.dtype, w.dist, w.seed + g) for g, m in enumerate(w.Ms)]


def _draw(gen: torch.Generator, shape, dist: str, lo_hi: int = 8) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "ints":
        return torch.randint(-lo_hi, lo_hi + 1, shape, generator=gen).to(torch.float32)
    if dist == "ones":
        return torch.ones(shape, dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


# The OCP FP8 formats, as the library's own types (E4M3 without infinities).
FP8_TORCH = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _pad(x: torch.Tensor, ld_pad: int) -> torch.Tensor:
    if ld_pad == 0:
        return x
    rows, cols = x.shape
    big = torch.full((rows, cols + ld_pad), float("nan"), dtype=x.dtype)
    big[:, :cols] = x
    return big[:, :cols]


def make_operands(M: int, N: int, K: int, dtype: str, dist: str, seed: int,
                  lda_pad: int = 0, ldb_pad: int = 0, lo_hi: int = 8):
    """(A, B) as CPU torch tensors: float32 for fp32/tf32, bfloat16 for bf16, float16 for
    fp16, float8 for e4m3 / e5m2.

    The tensors may be views with a leading dimension larger than their width
    (``*_pad``); use ``.stride(0)`` for the leading dimension.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    a = _draw(gen, (M, K), dist, lo_hi)
    b = _draw(gen, (K, N), dist, lo_hi)
    if dtype == "bf16":
        a = a.to(torch.bfloat16)
        b = b.to(torch.bfloat16)
    elif dtype == "fp16":
        a = a.to(torch.float16)
        b = b.to(torch.float16)
    elif dtype in FP8_TORCH:
        a = a.to(FP8_TORCH[dtype])
        b = b.to(FP8_TORCH[dtype])
    elif dtype not in ("fp32", "tf32"):
        raise ValueError(f"unknown dtype {dtype!r}")
    return _pad(a, lda_pad), _pad(b, ldb_pad)


OUT_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def make_epilogue_inputs(M: int, N: int, out: str, seed: int, scale: float = 1.0):
    """(c_old, bias): an M x N old C in the output type and N FP32 bias values,
    both N(0, scale^2), from their own seeded CPU generator."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed) + 7919)
    c_old = (torch.randn((M, N), generator=gen, dtype=torch.float32) * scale).to(OUT_TORCH[out])
    bias = torch.randn((N,), generator=gen, dtype=torch.float32) * scale
    return c_old, bias


def workload_operands(w: Workload):
    return make_operands(w.M, w.N, w.K, w.dtype, w.dist, w.seed)


def as_oracle_array(t: torch.Tensor) -> np.ndarray:
    """A CPU tensor as the numpy array the oracle takes (float32, uint16 BF16/FP16
    bits, or uint8 FP8 bytes)."""
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in FP8_TORCH.values():
        return t.view(torch.uint8).numpy()
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"unsupported operand dtype {t.dtype}")
