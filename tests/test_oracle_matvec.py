"""Pins for the f64 reference product and the pass criterion."""
from fractions import Fraction

import numpy as np

import synth
from oracle import fp16, matvec


def test_exact_rational_bruteforce():
    d = synth.fp16_dense(5, 40, seed=4)
    x = synth.activations(3, 40, seed=4)
    w64 = fp16.decode_f64(d["w"])
    y = matvec.gemv(w64, x)
    b = matvec.abs_bound(w64, x)
    for t in range(3):
        for r in range(5):
            acc = sum(Fraction(float(d["w"][r, c])) * Fraction(float(x[t, c])) for c in range(40))
            ab = sum(abs(Fraction(float(d["w"][r, c])) * Fraction(float(x[t, c]))) for c in range(40))
            assert abs(y[t, r] - float(acc)) <= 1e-14 * float(ab)
            assert abs(b[t, r] - float(ab)) <= 1e-14 * float(ab)


def test_unit_vectors_select_columns():
    d = synth.fp16_dense(7, 16, seed=8)
    x = np.eye(16, dtype=np.float16)
    y = matvec.gemv(fp16.decode_f64(d["w"]), x)
    assert np.array_equal(y, d["w"].astype(np.float64).T)      # token j gives column j


def test_pass_criterion():
    yref = np.array([[1.0, -2.0]])
    bound = np.array([[10.0, 100.0]])
    assert matvec.passes(yref, yref, bound).all()
    assert matvec.passes(yref + [[0.019, 0.19]], yref, bound).all()
    assert not matvec.passes(yref + [[0.021, 0.0]], yref, bound)[0, 0]
