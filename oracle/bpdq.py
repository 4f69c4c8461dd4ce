"""BPDQ decode, as the format is stated on "Qwen3-8B -- 2-bit BPDQ (packed)",
section Format:

    w[r, c] = sum_i coeffs[g(c), r, i] * bit_i(r, c) + coeffs[g(c), r, msbits]

with two bit-planes (i = 0, 1), group size 256 along the input dimension
(g(c) = c // 256) and one fp16 coefficient set (c0, c1, offset) per
(group, output row).  The "per-group offset" of the same section is read as
the third coefficient of the (group, row) set, which is what the formula
indexes.

Test infrastructure only (see ``oracle/__init__.py``).
"""
from __future__ import annotations

import numpy as np

GROUP = 256


def unpack_plane(plane: np.ndarray, C: int) -> np.ndarray:
    """uint8 [R][C/8] (bit i of byte j = column 8j+i) -> uint8 [R][C] of 0/1."""
    bits = np.unpackbits(plane, axis=1, bitorder="little")
    return bits[:, :C]


def decode_f64(plane0: np.ndarray, plane1: np.ndarray, coef: np.ndarray) -> np.ndarray:
    """Exact f64 weights w64[r][c] = c0[g][r]*b0 + c1[g][r]*b1 + off[g][r].

    Every term is an fp16 value times 0 or 1, so the f64 sum of three fp16
    values is exact.
    """
    R = plane0.shape[0]
    C = plane0.shape[1] * 8
    b0 = unpack_plane(plane0, C).astype(np.float64)
    b1 = unpack_plane(plane1, C).astype(np.float64)
    g = np.arange(C) // GROUP                       # g(c)
    cf = coef.astype(np.float64)                    # [G][R][3]
    c0 = cf[g, :, 0].T                              # [R][C]
    c1 = cf[g, :, 1].T
    off = cf[g, :, 2].T
    assert c0.shape == (R, C)
    return c0 * b0 + c1 * b1 + off


def decode_fp16(plane0: np.ndarray, plane1: np.ndarray, coef: np.ndarray) -> np.ndarray:
    """Canonical decoded weight: one round-to-nearest-even of the exact sum."""
    return decode_f64(plane0, plane1, coef).astype(np.float16)


def codes(plane0: np.ndarray, plane1: np.ndarray) -> np.ndarray:
    """The 2-bit code of each weight, plane 0 as the low bit: b0 | b1 << 1."""
    C = plane0.shape[1] * 8
    return unpack_plane(plane0, C) | (unpack_plane(plane1, C) << 1)
