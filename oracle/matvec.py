"""Reference product and pass criterion.

Every source page states the operation as y = W x for the packed W, one
call per projection (e.g. "Unfolding the Leech Lattice", introduction: a
fused dequantize-plus-matvec; every output row is verified against an f64
reference before any timing).  For N tokens x is [N][C] and y is [N][R]:

    y_ref[t][r] = sum_c w64[r][c] * x[t][c]          (f64)

An output passes when |y - y_ref| <= tol * sum_c |w64[r][c] * x[t][c]|, with
tol = 2e-3 for fp32 accumulation and an fp16 result.

Test infrastructure only (see ``oracle/__init__.py``).
"""
from __future__ import annotations

import numpy as np

TOL = 2e-3


def gemv(w64: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y_ref [N][R] in f64 (the library product is one step of the definition)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w64, dtype=np.float64).T


def abs_bound(w64: np.ndarray, x: np.ndarray) -> np.ndarray:
    """sum_c |w64[r][c] * x[t][c]| as [N][R]."""
    return np.abs(np.asarray(x, dtype=np.float64)) @ np.abs(np.asarray(w64, dtype=np.float64)).T


def passes(y: np.ndarray, y_ref: np.ndarray, bound: np.ndarray, tol: float = TOL) -> np.ndarray:
    err = np.abs(np.asarray(y, dtype=np.float64) - y_ref)
    return err <= tol * bound


def relative_error(y: np.ndarray, y_ref: np.ndarray, bound: np.ndarray) -> np.ndarray:
    err = np.abs(np.asarray(y, dtype=np.float64) - y_ref)
    return err / np.maximum(bound, np.finfo(np.float64).tiny)
