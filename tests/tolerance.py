"""Parity tolerance of the GEMM tests.

Fused epilogue (out = act(alpha A.B + beta C + bias), oracle/epilogue.py): the
product's bound scales by |alpha|, and the fp32 epilogue arithmetic (a multiply,
a fused multiply-add, an add; ReLU is exact and 1-Lipschitz) adds at most
2^-22 T with T = |alpha| S + |beta C| + |bias|, before the final rounding.

fp16/bf16 inputs (tensor-core path), any output format:
    |C_gpu - C_ref| <= 2^-10 * S + ulp_out(C_ref) / 2
fp32 inputs (SIMT path):
    |C_gpu - C_ref| <= 2^-20 * S
with C_ref the double-precision oracle and S[i,j] = sum_k |A[i,k] B[k,j]|.
The half ulp covers the final round-to-nearest into the output format;
ulp_out(x) = 2^(max(floor(log2|x|), e_min) - p + 1).  A finite C_ref must come
back finite.
"""
import numpy as np

# precision p (with hidden bit) and minimum normal exponent of each output format
_FMT = {"f16": (11, -14), "bf16": (8, -126), "f32": (24, -126)}


def ulp(x: np.ndarray, fmt: str) -> np.ndarray:
    p, emin = _FMT[fmt]
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(x > 0, x, 1.0))
    lead = np.where(x > 0, e - 1, emin)
    return np.ldexp(1.0, np.maximum(lead, emin) - p + 1)


def bound(C_ref: np.ndarray, S: np.ndarray, in_fmt: str, out_fmt: str) -> np.ndarray:
    if in_fmt == "f32":
        return 2.0 ** -20 * S
    return 2.0 ** -10 * S + 0.5 * ulp(C_ref, out_fmt)


def bound_epilogue(Z_ref: np.ndarray, S: np.ndarray, T: np.ndarray, alpha: float, in_fmt: str,
                   out_fmt: str) -> np.ndarray:
    core = 2.0 ** -20 * S if in_fmt == "f32" else 2.0 ** -10 * S
    return abs(alpha) * core + 2.0 ** -22 * T + 0.5 * ulp(Z_ref, out_fmt)


def check(C_gpu: np.ndarray, C_ref: np.ndarray, S: np.ndarray, in_fmt: str, out_fmt: str, tol=None):
    """Returns (ok, worst error/bound ratio, index of the worst element or None);
    `tol` replaces the product bound (e.g. bound_epilogue)."""
    C_gpu = np.asarray(C_gpu, dtype=np.float64)
    if tol is None:
        tol = bound(C_ref, S, in_fmt, out_fmt)
    finite_ref = np.isfinite(C_ref)
    bad_finite = finite_ref & ~np.isfinite(C_gpu)
    err = np.where(finite_ref, np.abs(C_gpu - C_ref), 0.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / tol, np.where(err > 0, np.inf, 0.0))
    ratio = np.where(bad_finite, np.inf, ratio)
    if ratio.size == 0:
        return True, 0.0, None
    worst = int(np.argmax(ratio))
    r = float(ratio.flat[worst])
    return bool(r <= 1.0), r, np.unravel_index(worst, ratio.shape)
