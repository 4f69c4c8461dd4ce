"""Pins for the Leech-lattice oracle and the lattice-point generator.

Page facts ("Unfolding the Leech Lattice", introduction): the ball of
shells up to 12 has 301 coordinate-permutation classes and about 1.1e14
points, named by a 47-bit index.  Classical facts (Conway and Sloane, cited
in section 7): the Golay weight enumerator, the kissing number 196560 and
the theta series.
"""
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import leech, matvec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golay_weight_enumerator():
    g = json.load(open(os.path.join(GOLDEN, "classical_lattice_facts.json")))
    assert leech.weight_enumerator() == {int(k): v for k, v in g["golay_weight_enumerator"].items()}
    # the generator's copy of the code is the same set of words
    a = {tuple(r) for r in leech.golay_code().tolist()}
    b = {tuple(r) for r in synth.golay_codewords().tolist()}
    assert a == b


def test_kissing_number_and_shell2_shapes():
    g = json.load(open(os.path.join(GOLDEN, "classical_lattice_facts.json")))
    assert leech.shell_size(2) == g["kissing_number"]
    assert sum(g["shell2_shapes"].values()) == g["kissing_number"]
    assert leech.shell_size(1) == 0


def test_page_ball_facts():
    g = json.load(open(os.path.join(GOLDEN, "leech_page_facts.json")))
    n = leech.ball_size(g["ball_shell_max"])
    assert abs(n - g["points_approx"]) <= g["points_rel_tolerance"] * g["points_approx"]
    assert n < 2 ** g["index_bits"] and n > 2 ** (g["index_bits"] - 1)
    assert len(leech.classes(1, g["ball_shell_max"])) == g["classes"]


def test_membership_rule_on_known_points():
    v = np.zeros(24, dtype=np.int64)
    v[[0, 5]] = [4, -4]
    assert leech.in_lattice(v) and leech.norm(v) == 32
    odd = np.ones(24, dtype=np.int64)
    odd[0] = -3
    assert leech.in_lattice(odd) and leech.norm(odd) == 32
    bad = odd.copy()
    bad[1] = -1                     # sum moves by 2 mod 8: not in the lattice
    assert not leech.in_lattice(bad)
    cw = leech.golay_code()[leech.golay_code().sum(axis=1) == 8][0]
    e = 2 * cw.astype(np.int64)
    assert leech.in_lattice(e)
    e[np.nonzero(cw)[0][0]] *= -1   # one minus sign: sum(z) odd
    assert not leech.in_lattice(e)


def test_generator_counts_match_theta_series():
    for m in range(2, 7):
        assert int(sum(synth.leech_shell_counts(m).values())) == leech.shell_size(m)


def test_generated_points_are_lattice_points_of_their_shell():
    d = synth.leech(16, 24 * 20 + 8, seed=3000)
    v, shell = d["v"].astype(np.int64), d["shell"]
    assert v.shape == (16, 20, 24)
    assert d["tail"].shape == (16, 8)
    assert shell.min() >= 2 and shell.max() <= 6
    for r in range(16):
        for b in range(20):
            assert leech.norm(v[r, b]) == 16 * shell[r, b]
            assert leech.in_lattice(v[r, b])


def test_generator_is_uniform_within_shell2():
    """Shell-2 shapes appear in proportion to their point counts."""
    rng = np.random.default_rng(123)
    n = 60000
    pts = synth._sample_shell(rng, np.full(n, 2))
    a = np.sort(np.abs(pts.astype(np.int64)), axis=1)[:, ::-1]
    twos = np.all(a[:, :8] == 2, axis=1) & np.all(a[:, 8:] == 0, axis=1)
    odds = (a[:, 0] == 3) & np.all(a[:, 1:] == 1, axis=1)
    fours = np.all(a[:, :2] == 4, axis=1) & np.all(a[:, 2:] == 0, axis=1)
    assert np.all(twos | odds | fours)
    for frac, cnt in ((twos.mean(), 97152), (odds.mean(), 98304), (fours.mean(), 1104)):
        p = cnt / 196560
        assert abs(frac - p) <= 5 * math.sqrt(p * (1 - p) / n)


def test_decode_closed_form():
    v = np.zeros((1, 1, 24), dtype=np.int8)
    v[0, 0, [0, 5]] = [4, -4]
    scale = np.array([0.5], dtype=np.float16)
    tail = np.array([[0.25, -1.0]], dtype=np.float16)
    w = leech.decode_f64(v, scale, tail)
    assert w.shape == (1, 26)
    assert w[0, 0] == pytest.approx(0.5 * 4 / math.sqrt(8), rel=1e-15)
    assert w[0, 5] == pytest.approx(-0.5 * 4 / math.sqrt(8), rel=1e-15)
    assert np.all(w[0, [1, 2, 3, 4] + list(range(6, 24))] == 0)
    assert w[0, 24] == 0.25 and w[0, 25] == -1.0
    x = np.zeros((1, 26), dtype=np.float16)
    x[0, 24] = 2.0                                  # only the tail contributes
    assert matvec.gemv(w, x)[0, 0] == 0.5
