"""Leech-lattice blocks ("Unfolding the Leech Lattice", introduction: weights
are grouped in blocks of 24 and each block is a point of the Leech lattice;
section 7: the lattice and its Golay construction are classical, after
Conway and Sloane).

The weight of column 24b + i of row r is scale_r * v_i / sqrt(8), where v is
the block's lattice point in integer coordinates (squared norm 16m for shell
m); columns past the last whole block form an unquantised fp16 tail
("Tetra", section 5.1: the kernel applies the row scale after the block dot
product and adds the unquantised tail).

Besides the decode, this module holds the lattice facts that pin the
generated inputs and this module itself: the binary Golay code, the
membership rule, the shell sizes from the theta series, and the count of
coordinate-permutation classes of the ball of shells up to 12 (the page
states 301 classes and 1.1e14 points named by a 47-bit index).

Test infrastructure only (see ``oracle/__init__.py``).
"""
from __future__ import annotations

import math
from functools import lru_cache

import numpy as np

BLOCK = 24


# ---------------------------------------------------------------- Golay code
@lru_cache(maxsize=1)
def golay_code() -> np.ndarray:
    """The extended quadratic-residue code of length 24 as int8 [4096][24].

    The length-23 quadratic-residue code is spanned by the all-ones word and
    the 23 cyclic shifts of the indicator of {0} and the quadratic residues
    modulo 23; coordinate 23 is an overall parity bit.  Row reduction over
    GF(2) gives a 12-row basis, whose 2^12 combinations are the code.
    """
    residues = {(i * i) % 23 for i in range(1, 23)}
    base = np.zeros(23, dtype=np.uint8)
    base[0] = 1
    base[list(residues)] = 1
    rows = [np.roll(base, j) for j in range(23)] + [np.ones(23, dtype=np.uint8)]
    M = np.array(rows, dtype=np.uint8)
    # Gaussian elimination over GF(2)
    basis = []
    col = 0
    M = M.copy()
    r = 0
    for col in range(23):
        piv = [i for i in range(r, M.shape[0]) if M[i, col]]
        if not piv:
            continue
        M[[r, piv[0]]] = M[[piv[0], r]]
        for i in range(M.shape[0]):
            if i != r and M[i, col]:
                M[i] ^= M[r]
        r += 1
    basis = M[:r]
    assert basis.shape[0] == 12, basis.shape
    coeffs = ((np.arange(4096)[:, None] >> np.arange(12)[None, :]) & 1).astype(np.uint8)
    words23 = (coeffs @ basis) % 2
    parity = words23.sum(axis=1) % 2
    return np.concatenate([words23, parity[:, None]], axis=1).astype(np.int8)


@lru_cache(maxsize=1)
def _codeword_set() -> frozenset:
    code = golay_code()
    return frozenset(int("".join(str(int(b)) for b in row[::-1]), 2) for row in code)


def is_codeword(bits: np.ndarray) -> bool:
    key = int("".join(str(int(b)) for b in np.asarray(bits)[::-1]), 2)
    return key in _codeword_set()


def weight_enumerator() -> dict:
    w = golay_code().sum(axis=1)
    vals, counts = np.unique(w, return_counts=True)
    return {int(a): int(b) for a, b in zip(vals, counts)}


# ---------------------------------------------------------- membership rule
def in_lattice(v: np.ndarray) -> bool:
    """Classical test for v in Z^24 (Conway and Sloane's coordinates, scaled
    so the minimal squared norm is 32): all coordinates share a parity p;
    sum(v) = 4p (mod 8); and the positions where v = 2 (mod 4) when p = 0, or
    v = 3 (mod 4) when p = 1, form a Golay codeword."""
    v = np.asarray(v, dtype=np.int64)
    p = int(v[0] & 1)
    if np.any((v & 1) != p):
        return False
    if (int(v.sum()) - 4 * p) % 8 != 0:
        return False
    target = 2 if p == 0 else 3
    return is_codeword(((v % 4) == target).astype(np.int8))


def norm(v: np.ndarray) -> int:
    v = np.asarray(v, dtype=np.int64)
    return int((v * v).sum())


# ------------------------------------------------------------- theta series
def _ramanujan_tau(nmax: int) -> list:
    """tau(1..nmax) from Delta(q) = q * prod_{n>=1} (1 - q^n)^24."""
    poly = [0] * (nmax + 1)
    poly[0] = 1
    for n in range(1, nmax + 1):
        for _ in range(24):                        # multiply by (1 - q^n)
            for k in range(nmax, n - 1, -1):
                poly[k] -= poly[k - n]
    # Delta = q * poly, so tau(m) = poly[m - 1]
    return [None] + [poly[m - 1] for m in range(1, nmax + 1)]


def shell_size(m: int) -> int:
    """Number of lattice points of squared norm 16m (norm 2m in the scaling
    with minimal norm 4): 65520/691 * (sigma_11(m) - tau(m)) for m >= 1,
    the coefficients of the lattice's theta series; 1 for m = 0."""
    if m == 0:
        return 1
    sigma11 = sum(d ** 11 for d in range(1, m + 1) if m % d == 0)
    tau = _ramanujan_tau(m)[m]
    num = 65520 * (sigma11 - tau)
    assert num % 691 == 0
    return num // 691


def ball_size(mmax: int) -> int:
    return sum(shell_size(m) for m in range(mmax + 1))


# ------------------------------------------- coordinate-permutation classes
def _multisets(values, n, target):
    """Multisets of n entries from ``values`` whose squares sum to target."""
    values = sorted(values, reverse=True)

    def rec(i, left, rem):
        if left == 0:
            if rem == 0:
                yield ()
            return
        if i == len(values):
            return
        a = values[i]
        q = a * a
        maxc = left if q == 0 else min(left, rem // q)
        for c in range(maxc, -1, -1):
            for rest in rec(i + 1, left - c, rem - c * q):
                yield (a,) * c + rest

    yield from rec(0, n, target)


def _realisable(pattern) -> bool:
    """Whether some arrangement and signs of the absolute values ``pattern``
    give a lattice point (membership rule above)."""
    weights = (0, 8, 12, 16, 24)
    if pattern[0] % 2 == 0:
        k = sum(1 for a in pattern if a % 4 == 2)
        if k not in weights:
            return False
        if k > 0:
            return True            # a sign flip on a 2 mod 4 entry moves the sum by 4 mod 8
        return sum(pattern) % 8 == 0
    # odd: the set S of positions with v = 3 (mod 4) must be a codeword, and
    # once S is fixed every sign is forced; check the sum modulo 8
    by_res = {r: sum(1 for a in pattern if a % 8 == r) for r in (1, 3, 5, 7)}
    for k in weights:
        for s1 in range(by_res[1] + 1):
            for s3 in range(by_res[3] + 1):
                for s5 in range(by_res[5] + 1):
                    s7 = k - s1 - s3 - s5
                    if s7 < 0 or s7 > by_res[7]:
                        continue
                    # in S: a = 1 mod 4 -> v = -a, a = 3 mod 4 -> v = +a
                    # not in S: a = 1 mod 4 -> v = +a, a = 3 mod 4 -> v = -a
                    tot = (s1 * (-1) + s3 * 3 + s5 * (-5) + s7 * 7
                           + (by_res[1] - s1) * 1 + (by_res[3] - s3) * (-3)
                           + (by_res[5] - s5) * 5 + (by_res[7] - s7) * (-7))
                    if tot % 8 == 4:
                        return True
    return False


def classes(mmin: int, mmax: int) -> list:
    """Sorted absolute-value patterns (coordinate-permutation classes up to
    sign) that occur in shells mmin..mmax."""
    out = []
    for m in range(mmin, mmax + 1):
        target = 16 * m
        amax = int(math.isqrt(target))
        evens = [a for a in range(0, amax + 1, 2)]
        odds = [a for a in range(1, amax + 1, 2)]
        for vals in (evens, odds):
            for pat in _multisets(vals, BLOCK, target):
                if _realisable(pat):
                    out.append((m, pat))
    return out


# -------------------------------------------------------------------- decode
INV_SQRT8 = 1.0 / math.sqrt(8.0)


def decode_f64(v: np.ndarray, scale: np.ndarray, tail: np.ndarray) -> np.ndarray:
    """w64[r][24b + i] = scale_r * v[r][b][i] / sqrt(8); tail columns copied."""
    R, nb, _ = v.shape
    body = scale.astype(np.float64)[:, None] * v.reshape(R, nb * BLOCK).astype(np.float64) * INV_SQRT8
    return np.concatenate([body, tail.astype(np.float64)], axis=1)
