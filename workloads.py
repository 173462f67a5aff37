"""Seeded synthetic inputs for the dense GEMM workloads.

This module is shared by the tests and by ``bench.py``.  It draws random
numbers and rounds them to the storage format of a workload; it holds none of
the GEMM arithmetic.  Neither the oracle nor the CUDA library imports it: a
caller generates the raw storage bits here and hands the same bits to both.

Workloads (C[M,N] = A[M,K] . B[K,N], row-major, fp32 accumulation).  The shapes
follow the sizes the tiling pages discuss: 64^3 (the 2x2-tile example of
"CUDA tile", section 2.1), 1024^3 / 2048^3 / 4096^3 (the three autotune shapes
of "GPU Kernel 的 Tile、Grid、Wave 与 Launch Overhead") and 4096^3 fp16/bf16
(the A100 optimisation walk-through of "Tiling 策略与内存层次优化", section
"实战：GEMM Kernel 完整 Tiling 分析").  The ragged 1000x1500x4096 case exercises
partial tiles and the zero-fill rule of "CUDA tile", section 四.4.

Random stream: splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; constants as in Vigna's public
reference implementation).  Output i (i = 1, 2, ...) of a stream seeded with s
is mix(s + i * 0x9E3779B97F4A7C15).

* uniform[-1, 1):  (r >> 11) * 2^-52 - 1
* N(0, 1):         Box-Muller with u1, u2 in (0, 1] (u = ((r >> 11) + 1) * 2^-53),
                   n = sqrt(-2 ln u1) * cos(2 pi u2); one normal per pair of
                   draws (draws 2i+1 and 2i+2 feed element i)
* scaling:         the normal workloads divide by sqrt(K) in double
* rounding:        round-to-nearest-even from double to the storage format,
                   overflow to infinity, gradual underflow
* seed:            0x7E11ED00 + 16 * workload.seed_index + (0 for A, 1 for B)
"""
from __future__ import annotations

from dataclasses import dataclass
import math

import numpy as np

# dtype codes of the C ABI: (input format, output format)
F32, F16, BF16, BF16_F32OUT, F16_F32OUT = 0, 1, 2, 3, 4
DTYPE_NAMES = {F32: "f32", F16: "f16", BF16: "bf16",
               BF16_F32OUT: "bf16_f32out", F16_F32OUT: "f16_f32out"}
IN_FORMAT = {F32: "f32", F16: "f16", BF16: "bf16", BF16_F32OUT: "bf16", F16_F32OUT: "f16"}
OUT_FORMAT = {F32: "f32", F16: "f16", BF16: "bf16", BF16_F32OUT: "f32", F16_F32OUT: "f32"}

# (precision p incl. hidden bit, minimum normal exponent, maximum exponent, bytes)
FORMATS = {
    "f16": (11, -14, 15, 2),
    "bf16": (8, -126, 127, 2),
    "f32": (24, -126, 127, 4),
}

SEED_BASE = 0x7E11ED00
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: int
    dist: str          # "uniform" or "normal"
    seed_index: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def in_bytes(self) -> int:
        return FORMATS[IN_FORMAT[self.dtype]][3]

    @property
    def out_bytes(self) -> int:
        return FORMATS[OUT_FORMAT[self.dtype]][3]

    @property
    def compulsory_bytes(self) -> int:
        return (self.M * self.K + self.K * self.N) * self.in_bytes + self.M * self.N * self.out_bytes


WORKLOADS = [
    Workload("f32_64x64x64", 64, 64, 64, F32, "uniform", 0),
    Workload("f16_1024x1024x1024", 1024, 1024, 1024, F16, "normal", 1),
    Workload("bf16_2048x2048x2048", 2048, 2048, 2048, BF16, "uniform", 2),
    Workload("bf16_4096x4096x4096_f32out", 4096, 4096, 4096, BF16_F32OUT, "normal", 3),
    Workload("bf16_1000x1500x4096_ragged", 1000, 1500, 4096, BF16, "uniform", 4),
    # fp32 shapes large enough to load the FP32 pipe
    Workload("f32_4096x4096x4096", 4096, 4096, 4096, F32, "uniform", 5),
    Workload("f32_2048x2048x2048", 2048, 2048, 2048, F32, "uniform", 6),
    # the two shapes "GPU Kernel 的 Tile、Grid、Wave 与 Launch Overhead" sets as exercises
    # (too few tiles to fill the GPU, and so many that the tile count must shrink)
    Workload("f16_512x512x512", 512, 512, 512, F16, "normal", 7),
    Workload("f16_8192x8192x8192", 8192, 8192, 8192, F16, "normal", 8),
]
BY_NAME = {w.name: w for w in WORKLOADS}


@dataclass(frozen=True)
class TransposeWorkload:
    """out = in^T for an in matrix of rows x cols ("CUDA tile", section 三),
    elements of elem_bytes moved as raw bits; inputs are seeded random bits."""
    name: str
    rows: int
    cols: int
    elem_bytes: int
    seed: int

    @property
    def bytes_moved(self) -> int:
        return 2 * self.rows * self.cols * self.elem_bytes


# Far larger than L2 (1 GiB per matrix for fp32), so every step streams HBM.
TRANSPOSE_WORKLOADS = [
    TransposeWorkload("transpose_f32_16384x16384", 16384, 16384, 4, 0x7A05E000),
    TransposeWorkload("transpose_bf16_16384x16384", 16384, 16384, 2, 0x7A05E001),
]
TRANSPOSE_BY_NAME = {w.name: w for w in TRANSPOSE_WORKLOADS}
HEADLINE = BY_NAME["bf16_4096x4096x4096_f32out"]


@dataclass(frozen=True)
class BatchWorkload:
    """A strided batch of `batch` products of one shape ("矩阵乘法中的平铺",
    closing advice on batched interfaces): matrix b of A is rows
    [b M, (b + 1) M) of one (batch M) x K array, of B rows [b K, (b + 1) K) of
    one (batch K) x N array, of C rows [b M, (b + 1) M) of (batch M) x N."""
    name: str
    batch: int
    M: int
    N: int
    K: int
    dtype: int
    dist: str
    seed_index: int

    @property
    def flops(self) -> int:
        return 2 * self.batch * self.M * self.N * self.K

    def one(self) -> Workload:
        """One product of the batch, as a workload (for checks and samples)."""
        return Workload(self.name + "_one", self.M, self.N, self.K, self.dtype, self.dist, self.seed_index)


# 64 products of 512^3: each alone fills 4 of 76 CTA pairs; the batch fills them all
BATCH_WORKLOADS = [BatchWorkload("batch64_bf16_512x512x512", 64, 512, 512, 512, BF16, "uniform", 9)]
BATCH_BY_NAME = {w.name: w for w in BATCH_WORKLOADS}


def make_batch_inputs(w: BatchWorkload):
    """(A_bits, B_bits): (batch M) x K and (batch K) x N, each from one seeded stream."""
    fmt = IN_FORMAT[w.dtype]
    A = make_matrix(w.batch * w.M, w.K, fmt, w.dist, seed_for(w.seed_index, "A"), w.K, None)
    B = make_matrix(w.batch * w.K, w.N, fmt, w.dist, seed_for(w.seed_index, "B"), w.K, None)
    return A, B


def seed_for(seed_index: int, which: str) -> int:
    return SEED_BASE + 16 * seed_index + (0 if which == "A" else 1)


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start+1 .. start+n of the splitmix64 stream seeded with ``seed``."""
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def uniform_pm1(seed: int, n: int) -> np.ndarray:
    r = splitmix64(seed, n)
    return (r >> np.uint64(11)).astype(np.float64) * 2.0 ** -52 - 1.0


def normal01(seed: int, n: int) -> np.ndarray:
    r = splitmix64(seed, 2 * n)
    u = ((r >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def round_to_format(x: np.ndarray, fmt: str) -> np.ndarray:
    """Round doubles to the nearest value of ``fmt`` (ties to even), as doubles.

    Magnitudes at or above the overflow threshold (max + half an ulp) become
    infinity; values below the smallest normal are rounded on the subnormal
    grid.  NaN stays NaN.
    """
    p, emin, emax, _ = FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0)
    xf = x[finite]
    _, e = np.frexp(xf)            # xf = m * 2^e, 0.5 <= |m| < 1
    exp = np.maximum(e - 1, emin)  # exponent of the leading bit, clamped to the subnormal range
    quantum = np.ldexp(1.0, exp - (p - 1))
    r = np.rint(xf / quantum) * quantum   # xf / quantum is exact (power-of-two scale); rint is ties-to-even
    max_val = (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
    r = np.where(np.abs(r) > max_val, np.copysign(np.inf, xf), r)
    out[finite] = r
    return out


def encode(x_rounded: np.ndarray, fmt: str) -> np.ndarray:
    """Storage bits of values already representable in ``fmt``."""
    if fmt == "f32":
        return x_rounded.astype(np.float32).view(np.uint32)
    if fmt == "f16":
        return x_rounded.astype(np.float16).view(np.uint16)
    if fmt == "bf16":
        b32 = x_rounded.astype(np.float32).view(np.uint32)
        return (b32 >> np.uint32(16)).astype(np.uint16)
    raise ValueError(fmt)


def decode(bits: np.ndarray, fmt: str) -> np.ndarray:
    """Storage bits -> float64 (exact)."""
    if fmt == "f32":
        return bits.view(np.float32).astype(np.float64)
    if fmt == "f16":
        return bits.view(np.float16).astype(np.float64)
    if fmt == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(fmt)


def draw(dist: str, seed: int, n: int, K: int) -> np.ndarray:
    if dist == "uniform":
        return uniform_pm1(seed, n)
    if dist == "normal":
        return normal01(seed, n) / math.sqrt(K)
    raise ValueError(dist)


def make_matrix(rows: int, cols: int, fmt: str, dist: str, seed: int, K: int, ld: int | None = None) -> np.ndarray:
    """A rows x cols matrix of storage bits, row-major with leading dimension ``ld``.

    Elements in the padding columns (ld > cols) are set to a NaN pattern so that
    a kernel that reads them poisons its output.
    """
    ld = cols if ld is None else ld
    vals = round_to_format(draw(dist, seed, rows * cols, K), fmt)
    bits = encode(vals, fmt).reshape(rows, cols)
    if ld == cols:
        return bits
    nan_bits = {"f32": 0x7FC00000, "f16": 0x7E00, "bf16": 0x7FC0}[fmt]
    out = np.full((rows, ld), nan_bits, dtype=bits.dtype)
    out[:, :cols] = bits
    return out


def make_inputs(w: Workload, lda: int | None = None, ldb: int | None = None):
    """(A_bits, B_bits) for workload ``w``."""
    fmt = IN_FORMAT[w.dtype]
    A = make_matrix(w.M, w.K, fmt, w.dist, seed_for(w.seed_index, "A"), w.K, lda)
    B = make_matrix(w.K, w.N, fmt, w.dist, seed_for(w.seed_index, "B"), w.K, ldb)
    return A, B


def small_integer_matrix(rows: int, cols: int, seed: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """Small integers (exact in every storage format), as float64."""
    r = splitmix64(seed, rows * cols)
    span = np.uint64(hi - lo + 1)
    return ((r % span).astype(np.int64) + lo).astype(np.float64).reshape(rows, cols)
