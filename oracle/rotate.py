"""Activation rotation ("Qwen3.8-27B on a 12 GB card", section "What the
kernel does per token"): the weights are stored in a rotated basis, so each
input is rotated at run time,

    x_rot = (H (x) Q) (S x),

with S a diagonal of random signs, H a Walsh-Hadamard transform of nh points
(the page names 1024 and 2048) and Q a small orthogonal nq x nq matrix,
C = nh * nq (the page's examples: 5120 = 5 x 1024, 6144 = 3 x 2048,
17408 = 17 x 1024).

Readings (the page leaves these open):
  * H is the orthonormal Sylvester Hadamard matrix, H[i][j] =
    (-1)^popcount(i & j) / sqrt(nh), so the rotation is orthogonal and W x =
    (W R^T)(R x) for the stored W R^T;
  * "(x)" is the Kronecker product in its usual index order: entry
    (i*nq + a, j*nq + b) of H (x) Q is H[i][j] * Q[a][b], so Q mixes each
    run of nq consecutive columns and H mixes the runs;
  * the sign of column c is bit c % 8 of byte c // 8 of ``signs``
    (1 = negate), the order the other packed planes use;
  * nh is 2048 when 2048 divides C, else 1024 (``default_split``), which
    reproduces the page's three examples.

The transform below follows the definition step by step: signs, then Q on
every run of nq columns, then the Walsh-Hadamard butterflies across runs,
then the 1/sqrt(nh) normalisation, all in f64.

Test infrastructure only (see ``oracle/__init__.py``).
"""
from __future__ import annotations

import numpy as np


def default_split(C: int) -> tuple[int, int]:
    """(nh, nq) with nh = 2048 if 2048 divides C, else 1024."""
    nh = 2048 if C % 2048 == 0 else 1024
    if C % nh:
        raise ValueError(f"C = {C} is not a multiple of {nh}")
    return nh, C // nh


def sign_vector(signs: np.ndarray, C: int) -> np.ndarray:
    """uint8 bitmask [C/8] -> f64 [C] of +1 / -1 (bit set = -1)."""
    bits = np.unpackbits(np.asarray(signs, dtype=np.uint8), bitorder="little")[:C]
    return 1.0 - 2.0 * bits.astype(np.float64)


def wht_f64(u: np.ndarray, axis: int) -> np.ndarray:
    """Unnormalised Sylvester Walsh-Hadamard transform along ``axis``:
    out[i] = sum_j (-1)^popcount(i & j) u[j], by the radix-2 butterflies
    (a, b) -> (a + b, a - b) on index pairs differing in one bit."""
    u = np.moveaxis(np.array(u, dtype=np.float64), axis, -1)
    n = u.shape[-1]
    if n & (n - 1):
        raise ValueError("Walsh-Hadamard length must be a power of two")
    h = 1
    while h < n:
        v = u.reshape(u.shape[:-1] + (n // (2 * h), 2, h))
        a, b = v[..., 0, :].copy(), v[..., 1, :].copy()
        v[..., 0, :] = a + b
        v[..., 1, :] = a - b
        u = v.reshape(u.shape)
        h *= 2
    return np.moveaxis(u, -1, axis)


def rotate_f64(x: np.ndarray, signs: np.ndarray, q: np.ndarray, nh: int) -> np.ndarray:
    """x_rot = (H (x) Q)(S x) in f64 for x [ntok][C] (any float dtype)."""
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    ntok, C = x.shape
    q = np.asarray(q, dtype=np.float64).reshape(-1)
    nq = C // nh
    if nh * nq != C or q.size != nq * nq:
        raise ValueError("C must equal nh * nq and q must be nq x nq")
    z = x * sign_vector(signs, C)                       # S x
    z = z.reshape(ntok, nh, nq)                         # z[t, j, b] = (S x)[t, j*nq + b]
    u = z @ q.reshape(nq, nq).T                         # u[t, j, a] = sum_b Q[a][b] z[t, j, b]
    r = wht_f64(u, axis=1) / np.sqrt(nh)                # out[t, i, a] = sum_j H[i][j] u[t, j, a]
    return r.reshape(ntok, C)


def abs_bound(x: np.ndarray, signs: np.ndarray, q: np.ndarray, nh: int) -> np.ndarray:
    """Per-output bound sum over terms of |H[i][j] Q[a][b] x[j*nq + b]|
    = (1/sqrt(nh)) * sum_j sum_b |Q[a][b]| |x[t, j*nq + b]| (independent of i)."""
    x = np.abs(np.atleast_2d(np.asarray(x, dtype=np.float64)))
    ntok, C = x.shape
    nq = C // nh
    qa = np.abs(np.asarray(q, dtype=np.float64).reshape(nq, nq))
    colsum = x.reshape(ntok, nh, nq).sum(axis=1)        # [t, b]
    per_a = colsum @ qa.T / np.sqrt(nh)                 # [t, a]
    return np.repeat(per_a[:, None, :], nh, axis=1).reshape(ntok, C)
