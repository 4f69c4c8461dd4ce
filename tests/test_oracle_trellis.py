"""Pins for the trellis oracle ("Qwen3.8-27B on a 12 GB card", section "A
trellis is a codebook you walk", and the worked packet of section "The
codebook is a hash").
"""
import json
import os

import numpy as np

import synth
from oracle import trellis

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_page_worked_packet_window():
    g = json.load(open(os.path.join(GOLDEN, "trellis_page_packet.json")))
    assert trellis.window(g["entry"], g["symbol"], g["T"], g["L"]) == g["state"]


def test_rate_is_T_over_V():
    assert trellis.stream_bits_per_weight() == 2.0
    d = synth.trellis(4, 512, seed=1)
    assert d["stream"].nbytes * 8 == 2 * 4 * 512


def _segment(sym):
    """A one-row, one-segment stream holding the 128 given symbols."""
    sym = np.asarray(sym, dtype=np.uint8)
    stream = (sym[0::2] | (sym[1::2] << 4)).astype(np.uint8)
    return stream.reshape(1, 1, 64)


def test_states_by_hand_with_wraparound():
    sym = np.zeros(128, dtype=np.uint8)
    sym[:4] = [1, 2, 3, 4]
    sym[125:] = [0xA, 0xB, 0xC]
    s = trellis.states(trellis.symbols(_segment(sym)))[0, 0]
    assert s[3] == 0x1234          # newest symbol in the low nibble
    assert s[0] == 0xABC1          # tail-biting: t125 t126 t127 t0
    assert s[1] == 0xBC12
    assert s[2] == 0xC123
    assert s[4] == 0x2340
    assert s[127] == 0x0ABC


def test_window_equals_state_recursion():
    d = synth.trellis(2, 512, seed=5)
    sym = trellis.symbols(d["stream"])
    s = trellis.states(sym)
    for r in range(2):
        for j in range(2):
            st = 0
            for k in range(125, 128):               # warm the state with the tail
                st = trellis.window(st, int(sym[r, j, k]), 4)
            for k in range(128):
                st = trellis.window(st, int(sym[r, j, k]), 4)
                assert st == s[r, j, k]


def test_index_hand_values_and_16_to_1():
    # ((s * 0x9E37) mod 2^32 & 0xFFFF) >> 4 evaluated by hand
    assert trellis.index(np.array([0]))[0] == 0
    assert trellis.index(np.array([1]))[0] == 0x9E3            # 0x9E37 >> 4
    assert trellis.index(np.array([2]))[0] == 0x3C6            # 0x13C6E & 0xFFFF = 0x3C6E
    assert trellis.index(np.array([0x10]))[0] == 0xE37         # 0x9E370 & 0xFFFF = 0xE370
    allidx = trellis.index(np.arange(1 << 16, dtype=np.uint32))
    counts = np.bincount(allidx, minlength=4096)
    assert counts.shape == (4096,) and np.all(counts == 16)


def test_sign_applies_to_both_weights():
    sym = np.zeros(128, dtype=np.uint8)
    sym[5] = 1                                   # s_5 = 0x0001: odd -> negative
    table = np.zeros((4096, 2), dtype=np.float16)
    table[0x9E3] = (1.5, -0.25)
    table[0] = (0.5, 2.0)
    u = trellis.decode_u(_segment(sym), table)[0]
    assert u[10] == -1.5 and u[11] == 0.25       # step 5 -> columns 10, 11
    # s_6 = 0x0010 -> index 0xE37 (zero row), s_4 = 0 -> index 0, positive
    assert u[8] == 0.5 and u[9] == 2.0


def test_decode_bit_serial_bruteforce():
    """Read the segment as a 512-bit little-endian stream, symbol k = bits
    4k..4k+3, and walk the state one symbol at a time."""
    d = synth.trellis(3, 512, seed=9)
    w = trellis.decode_f64(d["stream"], d["table"], d["scale"])
    for r in range(3):
        for j in range(2):
            bits = np.unpackbits(d["stream"][r, j], bitorder="little")
            syms = [int(sum(int(bits[4 * k + b]) << b for b in range(4))) for k in range(128)]
            for k in range(128):
                s = 0
                for age in (3, 2, 1, 0):
                    s = (s << 4) | syms[(k - age) % 128]
                idx = ((s * 0x9E37) % (1 << 32) & 0xFFFF) >> 4
                sg = -1.0 if s & 1 else 1.0
                for i in range(2):
                    expect = float(d["scale"][r]) * sg * float(d["table"][idx, i])
                    assert w[r, 256 * j + 2 * k + i] == expect


def test_fp32_canonical_is_exact():
    d = synth.trellis(4, 256, seed=2)
    w32 = trellis.decode_fp32(d["stream"], d["table"], d["scale"])
    w64 = trellis.decode_f64(d["stream"], d["table"], d["scale"])
    assert np.array_equal(w32.astype(np.float64), w64)
