"""Python access to the CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python binding
never do; the two share no code.

``oracle_gemm.c`` holds the arithmetic (a triple loop in double precision over
the decoded storage bits); this module compiles it with the host C compiler and
marshals numpy arrays.  ``perfmodel`` holds the pages' closed-form traffic,
intensity, occupancy and wave formulas.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle_gemm.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-pthread"]

# storage format codes of oracle_gemm.c
FMT = {"f32": 0, "f16": 1, "bf16": 2}
_lock = threading.Lock()
_lib = None


def compile_library(source: str = SOURCE, output: str = LIBRARY, extra: list[str] | None = None) -> str:
    """Compile an oracle source file into a shared library (gcc, no GPU needed)."""
    cmd = ["gcc", *CFLAGS, *(extra or []), "-o", output, source, "-lm"]
    subprocess.run(cmd, check=True)
    return output


def build() -> str:
    return compile_library()


def _stale() -> bool:
    return (not os.path.exists(LIBRARY)) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; returns a ctypes CDLL."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = _bind(ctypes.CDLL(LIBRARY))
    return _lib


def _bind(lib):
    i64, vp, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
    lib.oracle_gemm.argtypes = [i64, i64, i64, vp, i64, vp, i64, ip, dp, dp, ip]
    lib.oracle_gemm.restype = ip
    lib.oracle_gemm_blocked.argtypes = [i64, i64, i64, vp, i64, vp, i64, ip, dp, ip]
    lib.oracle_gemm_blocked.restype = ip
    lib.oracle_gemm_entries.argtypes = [i64, vp, i64, vp, i64, ip, i64, vp, vp, dp, dp]
    lib.oracle_gemm_entries.restype = None
    lib.oracle_decode.argtypes = [vp, ip, i64, i64, i64, dp]
    lib.oracle_decode.restype = None
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check_bits(X: np.ndarray, fmt: str):
    want = np.uint32 if fmt == "f32" else np.uint16
    if X.dtype != want or X.ndim != 2 or not X.flags.c_contiguous:
        raise ValueError(f"expected a C-contiguous 2-D {want.__name__} array of {fmt} bits")


def gemm(A: np.ndarray, B: np.ndarray, fmt: str, M: int, N: int, K: int,
         threads: int | None = None, with_abs: bool = True, lib=None):
    """Return (C, S) as float64 [M, N] arrays.

    A and B are 2-D arrays of storage bits whose row stride is their leading
    dimension (A: M x lda, lda >= K; B: K x ldb, ldb >= N).
    S[i, j] = sum_k |A[i, k] * B[k, j]| (None when ``with_abs`` is false).
    """
    lib = lib or load()
    _check_bits(A, fmt)
    _check_bits(B, fmt)
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if with_abs else None
    threads = threads or os.cpu_count() or 1
    rc = lib.oracle_gemm(M, N, K, _ptr(A), A.shape[1], _ptr(B), B.shape[1], FMT[fmt],
                         _ptr(C), _ptr(S) if S is not None else None, threads)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed: {rc}")
    return C, S


def gemm_blocked(A: np.ndarray, B: np.ndarray, fmt: str, M: int, N: int, K: int,
                 threads: int | None = None, lib=None) -> np.ndarray:
    lib = lib or load()
    _check_bits(A, fmt)
    _check_bits(B, fmt)
    C = np.zeros((M, N), dtype=np.float64)
    threads = threads or os.cpu_count() or 1
    rc = lib.oracle_gemm_blocked(M, N, K, _ptr(A), A.shape[1], _ptr(B), B.shape[1], FMT[fmt], _ptr(C), threads)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_blocked failed: {rc}")
    return C


def entries(A: np.ndarray, B: np.ndarray, fmt: str, K: int, rows, cols, lib=None):
    """(C, S) at the listed (row, col) positions, each computed independently."""
    lib = lib or load()
    _check_bits(A, fmt)
    _check_bits(B, fmt)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = rows.size
    c = np.zeros(n, dtype=np.float64)
    s = np.zeros(n, dtype=np.float64)
    lib.oracle_gemm_entries(K, _ptr(A), A.shape[1], _ptr(B), B.shape[1], FMT[fmt], n,
                            _ptr(rows), _ptr(cols), _ptr(c), _ptr(s))
    return c, s


def decode(X: np.ndarray, fmt: str, lib=None) -> np.ndarray:
    """The oracle's own decoding of storage bits into float64."""
    lib = lib or load()
    _check_bits(X, fmt)
    out = np.zeros(X.shape, dtype=np.float64)
    lib.oracle_decode(_ptr(X), FMT[fmt], X.shape[0], X.shape[1], X.shape[1], _ptr(out))
    return out
