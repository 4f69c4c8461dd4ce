"""Bitshift-trellis decode ("Qwen3.8-27B on a 12 GB card", section "A trellis
is a codebook you walk"): the state is L bits; each step shifts T new bits
in and emits V weights, so the rate is T/V bits per weight; in a bitshift
trellis the state is the last L bits of the stream, so position i is decoded
from one L-bit window, with no dependence between steps.

The configuration implemented: L = 16, T = 4, V = 2 (the page's V2T4 layout,
2 bits per weight).  The codebook is a shared table of 4096 x 2 fp16 values
indexed by ((s * 0x9E37) & 0xFFFF) >> 4; bit 0 of the state sets the sign of
both emitted weights (1 = negative); the stream restarts every 256 columns.

Readings (the pages leave these open):
  * the newest T bits are the least significant bits of the state (pinned
    by the page's worked packet, where entry byte 0x34 followed by symbol
    0x23 gives state 0x3423);
  * each 256-column segment is tail-biting: the window of step k reads
    symbols k-3 .. k modulo 128 inside the segment, which keeps the rate at
    exactly 2 bits per weight.

Test infrastructure only (see ``oracle/__init__.py``).
"""
from __future__ import annotations

import numpy as np

L, T, V = 16, 4, 2
SEGMENT = 256
STEPS = SEGMENT // V           # 128 steps per segment
HASH_MUL = 0x9E37


def window(prev_state: int, new_bits: int, t_bits: int, l_bits: int = L) -> int:
    """One trellis step: shift ``t_bits`` new bits into an ``l_bits`` state,
    newest bits least significant."""
    return ((prev_state << t_bits) | new_bits) & ((1 << l_bits) - 1)


def symbols(stream: np.ndarray) -> np.ndarray:
    """uint8 [R][S][64] -> uint8 [R][S][128]; symbol 2i is the low nibble of
    byte i, symbol 2i+1 its high nibble."""
    lo = stream & 0x0F
    hi = stream >> 4
    out = np.empty(stream.shape[:-1] + (STEPS,), dtype=np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def states(sym: np.ndarray) -> np.ndarray:
    """State of each step: s_k = t_{k-3}<<12 | t_{k-2}<<8 | t_{k-1}<<4 | t_k,
    indices modulo 128 inside the segment (tail-biting)."""
    t = sym.astype(np.uint32)
    s = np.zeros_like(t)
    for age in range(L // T):                      # age 0 = newest symbol
        s |= np.roll(t, age, axis=-1) << (T * age)
    return s


def index(s: np.ndarray) -> np.ndarray:
    """Table row of a state: ((s * 0x9E37) mod 2^32 & 0xFFFF) >> 4."""
    h = (s.astype(np.uint64) * HASH_MUL) & 0xFFFFFFFF
    return ((h & 0xFFFF) >> 4).astype(np.int64)


def sign(s: np.ndarray) -> np.ndarray:
    """+1 or -1: state bit 0 set means negative."""
    return np.where((s & 1) != 0, -1.0, 1.0)


def decode_u(stream: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Unscaled weights u[r][c] (fp16, exact): column 256j + 2k + i of row r is
    sign(s_k) * table[index(s_k)][i] for segment j, step k."""
    R, S = stream.shape[:2]
    s = states(symbols(stream))                    # [R][S][128]
    idx = index(s)
    sg = sign(s)
    tab = table.astype(np.float64)
    u = sg[..., None] * tab[idx]                   # [R][S][128][2]
    return u.reshape(R, S * SEGMENT).astype(np.float16)


def decode_f64(stream: np.ndarray, table: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Exact weights w64 = scale_r * u (a product of two fp16 values)."""
    u = decode_u(stream, table).astype(np.float64)
    return scale.astype(np.float64)[:, None] * u


def decode_fp32(stream: np.ndarray, table: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Canonical decoded weight: float(scale) * float(u) in fp32 (exact, since
    a product of two fp16 significands needs at most 22 bits)."""
    u = decode_u(stream, table).astype(np.float32)
    return scale.astype(np.float32)[:, None] * u


def stream_bits_per_weight() -> float:
    """Rate of the code: T / V bits per weight."""
    return T / V
