"""Fused epilogue of the oracle -- TEST INFRASTRUCTURE ONLY (same rules as the
rest of ``oracle/``: only ``tests/``, ``smoke()`` and ``bench.py``'s CPU legs
use it; the CUDA library never does).

"Tiling 策略与内存层次优化", section "Tiling 贯穿编译器栈" (its Fusion stage):
element-wise post-processing such as a bias add and ReLU is applied to a GEMM
tile's output in place, before the result goes back to memory (epilogue
fusion).  The pages give no formula; the reading taken here is the common one:
the bias is a per-column vector added before the activation, and the product
may be scaled and accumulated onto the prior C as in BLAS (alpha, beta):

    Z[i, j] = alpha * D[i, j] + beta * Cin[i, j] + bias[j]
    out[i, j] = 0 if Z[i, j] < 0 else Z[i, j]     (act = "relu")
              = Z[i, j]                           (act = "none")

D is the exact product from ``oracle.gemm``.  With beta == 0 the prior C is
not read at all, so whatever it holds (NaN included) has no effect.  ReLU keeps
a NaN (it is not below zero) and maps -0 to -0.  Everything is float64.
"""
from __future__ import annotations

import numpy as np

ACTS = ("none", "relu")


def apply(D: np.ndarray, Cin: np.ndarray | None = None, alpha: float = 1.0, beta: float = 0.0,
          bias: np.ndarray | None = None, act: str = "none") -> np.ndarray:
    """The epilogue on the exact product D (M x N); Cin (M x N) and bias (N)
    as float64 values (decoded storage)."""
    if act not in ACTS:
        raise ValueError(f"unknown activation {act!r}")
    D = np.asarray(D, dtype=np.float64)
    Z = alpha * D
    if beta != 0.0:
        Z = Z + beta * np.asarray(Cin, dtype=np.float64)
    if bias is not None:
        Z = Z + np.asarray(bias, dtype=np.float64)[None, :]
    if act == "relu":
        Z = np.where(Z < 0.0, 0.0, Z)
    return Z


def magnitude(S: np.ndarray, Cin: np.ndarray | None = None, alpha: float = 1.0, beta: float = 0.0,
              bias: np.ndarray | None = None) -> np.ndarray:
    """T = |alpha| S + |beta Cin| + |bias|: the size of the terms the epilogue
    adds, which sets the rounding error of doing it in fp32."""
    T = abs(alpha) * np.asarray(S, dtype=np.float64)
    if beta != 0.0:
        T = T + np.abs(beta * np.asarray(Cin, dtype=np.float64))
    if bias is not None:
        T = T + np.abs(np.asarray(bias, dtype=np.float64))[None, :]
    return T
