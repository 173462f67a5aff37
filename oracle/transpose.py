"""Tiled transpose of the oracle -- TEST INFRASTRUCTURE ONLY (same rules as the
rest of ``oracle/``: only ``tests/``, ``smoke()`` and ``bench.py``'s CPU legs
use it; the CUDA library never does).

"CUDA tile", section 三 (tiling beyond matrix multiply; the transpose example):
out[j][i] = in[i][j] for an in matrix of rows x cols, with rows of in stored
ld_in elements apart and rows of out ld_out elements apart.  Tiling only makes
both the reads and the writes coalesced; the result is the plain definition.
Elements are moved as raw storage units (bytes), so the result is bit-exact.
"""
from __future__ import annotations

import numpy as np


def transpose(src: np.ndarray, rows: int, cols: int, out: np.ndarray | None = None,
              ld_out: int | None = None) -> np.ndarray:
    """out (cols x ld_out, ld_out >= rows) with out[j, i] = src[i, j] for
    i < rows, j < cols; the columns of out past `rows` keep what `out` held."""
    if src.ndim != 2 or src.shape[0] < rows or src.shape[1] < cols:
        raise ValueError("src must be rows x ld_in with ld_in >= cols")
    ld_out = rows if ld_out is None else ld_out
    if ld_out < rows:
        raise ValueError("ld_out must be >= rows")
    if out is None:
        out = np.zeros((cols, ld_out), dtype=src.dtype)
    for j in range(cols):          # row j of out is column j of src
        out[j, :rows] = src[:rows, j]
    return out
