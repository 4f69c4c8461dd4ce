"""Seeded synthetic inputs for the packed 2-bit GEMV path.

This module is shared by the oracle (under ``oracle/``) and by the CUDA path
(``dequant_gemv_q2_gb300``).  It only draws random canonical arrays; it holds
none of the decode or matvec arithmetic, and it imports neither side.

Every generator uses numpy's PCG64 (``numpy.random.default_rng``) seeded with
a ``(seed, stream)`` tuple, draws in the order written in its docstring, and
rounds f64 draws to fp16 with round-to-nearest-even (numpy's ``astype``).

Canonical layouts (the arrays the packers take):

* BPDQ   -- ``plane0``, ``plane1``: uint8 ``[R][C/8]``; bit ``i`` (LSB first)
  of byte ``j`` is the plane bit of column ``8j+i``.  ``coef``: fp16
  ``[C/256][R][3]`` holding ``(c0, c1, off)`` per (group, row).
* trellis -- ``stream``: uint8 ``[R][C/256][64]``; byte ``i`` of a segment
  holds symbol ``2i`` in its low nibble and symbol ``2i+1`` in its high
  nibble.  ``table``: fp16 ``[4096][2]``.  ``scale``: fp16 ``[R]``.
* Leech  -- ``v``: int8 ``[R][C//24][24]`` lattice points in integer
  coordinates, ``shell``: int ``[R][C//24]``, ``tail``: fp16 ``[R][C%24]``,
  ``scale``: fp16 ``[R]``.
* fp16 dense -- ``w``: fp16 ``[R][C]``.
* activations -- ``x``: fp16 ``[N][C]``.
* rotation -- ``signs``: uint8 ``[ceil(C/8)]`` column sign bits, ``q``: fp32
  ``[nq][nq]`` orthogonal, C = nh * nq.
"""
from __future__ import annotations

import numpy as np

GROUP = 256          # BPDQ group size along the input dimension
SEGMENT = 256        # trellis restart interval in columns
BLOCK = 24           # Leech block length
TABLE_ENTRIES = 4096  # trellis codebook rows


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng((int(seed), int(stream)))


def activations(N: int, C: int, seed: int) -> np.ndarray:
    """x ~ N(0, 1) rounded to fp16, shape [N][C] (stream 1 of ``seed``)."""
    rng = _rng(seed, 1)
    return rng.normal(0.0, 1.0, size=(N, C)).astype(np.float16)


def bpdq(R: int, C: int, seed: int) -> dict:
    """BPDQ canonical weights.

    Draw order: plane0 bytes, plane1 bytes (uniform, i.e. uniform random
    bits), c0 ~ N(0, 0.02^2), c1 ~ N(0, 0.02^2), off ~ N(0, 0.01^2), each
    [G][R].
    """
    if C % GROUP:
        raise ValueError("BPDQ needs C % 256 == 0")
    G = C // GROUP
    rng = _rng(seed, 0)
    plane0 = rng.integers(0, 256, size=(R, C // 8), dtype=np.uint8)
    plane1 = rng.integers(0, 256, size=(R, C // 8), dtype=np.uint8)
    c0 = rng.normal(0.0, 0.02, size=(G, R))
    c1 = rng.normal(0.0, 0.02, size=(G, R))
    off = rng.normal(0.0, 0.01, size=(G, R))
    coef = np.stack([c0, c1, off], axis=-1).astype(np.float16)
    return {"R": R, "C": C, "plane0": plane0, "plane1": plane1, "coef": coef}


def trellis(R: int, C: int, seed: int) -> dict:
    """Bitshift-trellis canonical weights (L=16, T=4, V=2, 256-column restart).

    Draw order: the symbol stream as uniform bytes [R][C/256][64], the
    codebook table ~ N(0, 1) [4096][2], the row scale ~ U(0.005, 0.03) [R].
    """
    if C % SEGMENT:
        raise ValueError("trellis needs C % 256 == 0")
    rng = _rng(seed, 0)
    stream = rng.integers(0, 256, size=(R, C // SEGMENT, 64), dtype=np.uint8)
    table = rng.normal(0.0, 1.0, size=(TABLE_ENTRIES, 2)).astype(np.float16)
    scale = rng.uniform(0.005, 0.03, size=R).astype(np.float16)
    return {"R": R, "C": C, "stream": stream, "table": table, "scale": scale}


def fp16_dense(R: int, C: int, seed: int) -> dict:
    """Dense fp16 control weights ~ N(0, 0.02^2)."""
    rng = _rng(seed, 0)
    w = rng.normal(0.0, 0.02, size=(R, C)).astype(np.float16)
    return {"R": R, "C": C, "w": w}


# --------------------------------------------------------------------------
# Leech lattice points.  The sampler needs a binary Golay code to place the
# points; it uses the extended quadratic-residue code of length 24 (the
# length-23 code spanned by the all-ones word and the cyclic shifts of the
# indicator of {0} and the quadratic residues mod 23, plus an overall parity
# bit).  A point of shell m has squared norm 16m and is either
#   even: v = 2c + 4z with sum(z) even, or
#   odd:  v = 1 + 2c + 4z with sum(z) odd,
# for a codeword c and an integer vector z.
# --------------------------------------------------------------------------

def _golay_codewords() -> np.ndarray:
    qr = sorted({(i * i) % 23 for i in range(1, 23)})
    support = [0] + qr
    gens = [sum(1 << ((s + j) % 23) for s in support) for j in range(23)]
    gens.append((1 << 23) - 1)
    basis: list[int] = []
    for g in gens:
        v = g
        for b in basis:
            v = min(v, v ^ b)
        if v:
            basis.append(v)
            basis.sort(reverse=True)
    words = [0]
    for b in basis:
        words += [w ^ b for w in words]
    ext = [w | ((bin(w).count("1") & 1) << 23) for w in words]
    bits = np.array([[(w >> i) & 1 for i in range(24)] for w in sorted(ext)], dtype=np.int8)
    return bits


_GOLAY = None


def golay_codewords() -> np.ndarray:
    """All 4096 codewords of the code above as an int8 [4096][24] 0/1 array."""
    global _GOLAY
    if _GOLAY is None:
        _GOLAY = _golay_codewords()
    return _GOLAY


# per-coordinate options (v, z) for parity p and codeword bit c, |v| <= 9
def _options(p: int, c: int) -> list[tuple[int, int]]:
    out = []
    for z in range(-3, 4):
        v = p + 2 * c + 4 * z
        if abs(v) <= 9:
            out.append((v, z))
    return out


_MAXN = 16 * 6


def _count_tables() -> dict:
    """F[p][k1][k0][n][par]: ways to fill k1 coordinates with c=1 and k0 with
    c=0 (parity class p) so that the squared norm is n and sum(z) = par mod 2."""
    tabs = {}
    for p in (0, 1):
        F = np.zeros((25, 25, _MAXN + 1, 2), dtype=np.float64)
        F[0, 0, 0, 0] = 1.0
        for k1 in range(25):
            for k0 in range(25 - k1):
                if k1 == 0 and k0 == 0:
                    continue
                if k1 > 0:
                    prev, opts = F[k1 - 1, k0], _options(p, 1)
                else:
                    prev, opts = F[k1, k0 - 1], _options(p, 0)
                acc = np.zeros((_MAXN + 1, 2))
                for v, z in opts:
                    q = v * v
                    if q > _MAXN:
                        continue
                    par = z & 1
                    acc[q:, 0] += prev[: _MAXN + 1 - q, par]
                    acc[q:, 1] += prev[: _MAXN + 1 - q, 1 - par]
                F[k1, k0] = acc
        tabs[p] = F
    return tabs


_TABS = None


def leech_shell_counts(m: int) -> dict:
    """Number of lattice points of shell m by (parity class, codeword weight),
    from the sampler's own counting tables (used by the sampler and pinned
    against the theta series in the tests)."""
    global _TABS
    if _TABS is None:
        _TABS = _count_tables()
    cw = golay_codewords().sum(axis=1)
    out = {}
    for p in (0, 1):
        for w in (0, 8, 12, 16, 24):
            A = int((cw == w).sum())
            out[(p, w)] = A * _TABS[p][w, 24 - w, 16 * m, p]
    return out


def _sample_shell(rng: np.random.Generator, m: np.ndarray) -> np.ndarray:
    """Uniform lattice points within shell m[i] for each i (vectorised)."""
    global _TABS
    if _TABS is None:
        _TABS = _count_tables()
    cws = golay_codewords()
    wt = cws.sum(axis=1)
    B = m.shape[0]
    out = np.zeros((B, 24), dtype=np.int8)
    # 1. (parity class, codeword weight) in proportion to point counts
    keys = [(p, w) for p in (0, 1) for w in (0, 8, 12, 16, 24)]
    probs = np.zeros((7, len(keys)))
    for mm in range(2, 7):
        cnt = leech_shell_counts(mm)
        probs[mm] = np.array([cnt[k] for k in keys], dtype=np.float64)
        probs[mm] /= probs[mm].sum()
    u = rng.random(B)
    cum = np.cumsum(probs[m], axis=1)
    kidx = (u[:, None] >= cum).sum(axis=1)
    kidx = np.minimum(kidx, len(keys) - 1)
    par_cls = np.array([k[0] for k in keys])[kidx]
    weight = np.array([k[1] for k in keys])[kidx]
    # 2. a uniform codeword of that weight
    code = np.zeros((B, 24), dtype=np.int8)
    u2 = rng.random(B)
    for w in (0, 8, 12, 16, 24):
        sel = np.nonzero(weight == w)[0]
        if sel.size == 0:
            continue
        pool = cws[wt == w]
        pick = np.minimum((u2[sel] * pool.shape[0]).astype(np.int64), pool.shape[0] - 1)
        code[sel] = pool[pick]
    # 3. coordinates one by one from the suffix counts
    k1 = code.sum(axis=1).astype(np.int64)
    k0 = 24 - k1
    nrem = (16 * m).astype(np.int64)
    prem = par_cls.astype(np.int64)          # required parity of sum(z) left
    u3 = rng.random((24, B))
    for i in range(24):
        ci = code[:, i].astype(np.int64)
        nk1 = k1 - ci
        nk0 = k0 - (1 - ci)
        # candidate z in -3..3 (|v| <= 9 covers every shell up to m = 6)
        zs = np.arange(-3, 4)
        vals = par_cls[:, None] + 2 * ci[:, None] + 4 * zs[None, :]          # [B][7]
        q = vals * vals
        nn = nrem[:, None] - q
        ok = (np.abs(vals) <= 9) & (nn >= 0)
        nn_c = np.clip(nn, 0, _MAXN)
        pp = (prem[:, None] - zs[None, :]) & 1
        Fsel0 = _TABS[0][nk1[:, None], nk0[:, None], nn_c, pp]
        Fsel1 = _TABS[1][nk1[:, None], nk0[:, None], nn_c, pp]
        wts = np.where(par_cls[:, None] == 0, Fsel0, Fsel1) * ok
        cum = np.cumsum(wts, axis=1)
        tot = cum[:, -1:]
        pick = (u3[i][:, None] * tot >= cum).sum(axis=1)
        pick = np.minimum(pick, 6)
        v = vals[np.arange(B), pick]
        z = zs[pick]
        out[:, i] = v
        nrem = nrem - v * v
        prem = (prem - z) & 1
        k1, k0 = nk1, nk0
    return out


def leech(R: int, C: int, seed: int) -> dict:
    """Leech-lattice canonical weights.

    Each 24-column block of a row is a lattice point of a shell m drawn
    uniformly from {2..6}, uniform within the shell.  Draw order: shells
    [R][C//24], the point sampler's uniforms (class, codeword, then 24
    coordinates), the row scale ~ U(0.005, 0.03) [R], the dense tail
    ~ N(0, 0.01^2) [R][C%24].
    """
    nb = C // BLOCK
    rng = _rng(seed, 0)
    shell = rng.integers(2, 7, size=(R, nb))
    if R * nb:
        v = _sample_shell(rng, shell.reshape(-1)).reshape(R, nb, BLOCK)
    else:
        v = np.zeros((R, nb, BLOCK), dtype=np.int8)
    scale = rng.uniform(0.005, 0.03, size=R).astype(np.float16)
    tail = rng.normal(0.0, 0.01, size=(R, C % BLOCK)).astype(np.float16)
    return {"R": R, "C": C, "v": v, "shell": shell, "scale": scale, "tail": tail}


def rotation(C: int, nh: int, seed: int) -> dict:
    """Inputs of the activation rotation x_rot = (H (x) Q)(S x).

    Draw order: ``signs`` uint8 [ceil(C/8)] uniform bytes (bit c % 8 of byte
    c // 8 is the sign of column c, 1 = negate); then an nq x nq matrix of
    N(0, 1) draws, nq = C / nh, whose QR factor (numpy.linalg.qr, columns
    sign-fixed by the diagonal of R) is rounded to fp32 as ``q`` (row-major,
    orthogonal to fp32 rounding).
    """
    if C % nh:
        raise ValueError("C must be a multiple of nh")
    nq = C // nh
    rng = _rng(seed, 2)
    signs = rng.integers(0, 256, size=(C + 7) // 8, dtype=np.uint8)
    g = rng.normal(0.0, 1.0, size=(nq, nq))
    qm, rm = np.linalg.qr(g)
    qm = qm * np.sign(np.diag(rm))[None, :]
    return {"C": C, "nh": nh, "nq": nq, "signs": signs, "q": qm.astype(np.float32)}
