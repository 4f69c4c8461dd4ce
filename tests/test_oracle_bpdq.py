"""Pins for the BPDQ oracle ("Qwen3-8B -- 2-bit BPDQ (packed)", section Format).

The checks use closed forms and special cases of
w[r, c] = c0[g, r] * b0 + c1[g, r] * b1 + off[g, r], g = c // 256, and an
exact rational brute force, so that a swapped plane, a wrong group index, a
wrong bit order or a dropped offset fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import bpdq, matvec


def _coef(G, R, vals):
    coef = np.zeros((G, R, 3), dtype=np.float16)
    for (g, r), (c0, c1, off) in vals.items():
        coef[g, r] = (c0, c1, off)
    return coef


@pytest.fixture
def two_groups():
    # R = 2, C = 512: two groups with distinct, fp16-exact coefficients
    coef = _coef(2, 2, {(0, 0): (0.5, 0.25, -0.125), (0, 1): (-1.0, 2.0, 0.0625),
                        (1, 0): (0.75, -0.5, 0.25), (1, 1): (0.03125, 1.5, -2.0)})
    return coef


@pytest.mark.parametrize("b0,b1", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_closed_form_constant_planes(two_groups, b0, b1):
    R, C = 2, 512
    p0 = np.full((R, C // 8), 0xFF * b0, dtype=np.uint8)
    p1 = np.full((R, C // 8), 0xFF * b1, dtype=np.uint8)
    w = bpdq.decode_f64(p0, p1, two_groups)
    for r in range(R):
        for g in range(2):
            c0, c1, off = (float(v) for v in two_groups[g, r])
            expect = off + b0 * c0 + b1 * c1
            assert np.all(w[r, 256 * g:256 * (g + 1)] == expect)


def test_single_bit_lsb_first(two_groups):
    R, C = 2, 512
    for col in (0, 1, 7, 8, 255, 256, 300, 511):
        p0 = np.zeros((R, C // 8), dtype=np.uint8)
        p1 = np.zeros((R, C // 8), dtype=np.uint8)
        p0[1, col // 8] = 1 << (col % 8)          # row 1, plane 0 bit of column col
        w = bpdq.decode_f64(p0, p1, two_groups)
        g = col // 256
        c0, _, off = (float(v) for v in two_groups[g, 1])
        assert w[1, col] == off + c0
        others = np.delete(w[1], col)
        offs = np.where(np.delete(np.arange(C), col) < 256,
                        float(two_groups[0, 1, 2]), float(two_groups[1, 1, 2]))
        assert np.array_equal(others, offs)
        assert np.all(w[0] == np.repeat([float(two_groups[0, 0, 2]), float(two_groups[1, 0, 2])], 256))


def test_code_low_bit_is_plane0():
    p0 = np.array([[0b00000101]], dtype=np.uint8)
    p1 = np.array([[0b00000110]], dtype=np.uint8)
    # columns 0..3: (b0, b1) = (1,0), (0,1), (1,1), (0,0)
    assert bpdq.codes(p0, p1)[0, :4].tolist() == [1, 2, 3, 0]


def test_fp16_is_one_rounding_of_exact_sum():
    d = synth.bpdq(8, 512, seed=7)
    w16 = bpdq.decode_fp16(d["plane0"], d["plane1"], d["coef"])
    b0 = bpdq.unpack_plane(d["plane0"], 512)
    b1 = bpdq.unpack_plane(d["plane1"], 512)
    for r in range(8):
        for c in range(0, 512, 37):
            c0, c1, off = (Fraction(float(v)) for v in d["coef"][c // 256, r])
            exact = c0 * int(b0[r, c]) + c1 * int(b1[r, c]) + off
            assert w16[r, c] == np.float16(float(exact))   # exact fits f64; one rounding to fp16


def test_all_zero_planes_gives_offset_times_group_sums():
    R, C = 3, 768
    d = synth.bpdq(R, C, seed=11)
    z = np.zeros_like(d["plane0"])
    x = synth.activations(2, C, seed=11)
    y = matvec.gemv(bpdq.decode_f64(z, z, d["coef"]), x)
    xs = x.astype(np.float64).reshape(2, 3, 256).sum(axis=2)       # X_g per token
    off = d["coef"][:, :, 2].astype(np.float64)                     # [G][R]
    np.testing.assert_allclose(y, xs @ off, rtol=1e-12, atol=1e-12)


def test_exact_rational_bruteforce():
    R, C, N = 3, 256, 2
    d = synth.bpdq(R, C, seed=3)
    x = synth.activations(N, C, seed=3)
    y = matvec.gemv(bpdq.decode_f64(d["plane0"], d["plane1"], d["coef"]), x)
    for t in range(N):
        for r in range(R):
            acc = Fraction(0)
            for c in range(C):
                b0 = (int(d["plane0"][r, c // 8]) >> (c % 8)) & 1
                b1 = (int(d["plane1"][r, c // 8]) >> (c % 8)) & 1
                c0, c1, off = (Fraction(float(v)) for v in d["coef"][c // 256, r])
                acc += (c0 * b0 + c1 * b1 + off) * Fraction(float(x[t, c]))
            assert abs(y[t, r] - float(acc)) <= 1e-12 * max(1.0, abs(float(acc)))


def _closed_form_holds(decode, coef):
    R, C = 2, 512
    for b0, b1 in ((1, 0), (0, 1)):
        p0 = np.full((R, C // 8), 0xFF * b0, dtype=np.uint8)
        p1 = np.full((R, C // 8), 0xFF * b1, dtype=np.uint8)
        w = decode(p0, p1, coef)
        for r in range(R):
            for g in range(2):
                c0, c1, off = (float(v) for v in coef[g, r])
                if not np.all(w[r, 256 * g:256 * (g + 1)] == off + b0 * c0 + b1 * c1):
                    return False
    return True


def test_planted_mistakes_are_caught(two_groups, monkeypatch):
    """Mistakes planted in a copy of the oracle break the closed form."""
    assert _closed_form_holds(bpdq.decode_f64, two_groups)
    swapped = lambda p0, p1, coef: bpdq.decode_f64(p1, p0, coef)       # planes swapped
    assert not _closed_form_holds(swapped, two_groups)
    rolled = lambda p0, p1, coef: bpdq.decode_f64(p0, p1, coef[::-1])  # groups reversed
    assert not _closed_form_holds(rolled, two_groups)
