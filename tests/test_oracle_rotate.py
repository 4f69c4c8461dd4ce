"""Pins of the activation-rotation oracle (``oracle/rotate.py``) against
facts it does not compute itself: scipy's Hadamard construction, the
Sylvester closed form, a dense Kronecker product built with numpy.kron,
orthogonality (norms and the inverse), and the page's size examples
(``tests/golden/rotation_page_facts.json``: "Qwen3.8-27B on a 12 GB card",
section "What the kernel does per token")."""
import json
import os

import numpy as np
import pytest

import synth
from oracle import rotate

scipy_linalg = pytest.importorskip("scipy.linalg")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rotation_page_facts.json")


@pytest.mark.parametrize("n", [1, 2, 4, 8, 64, 256])
def test_wht_matches_scipy_hadamard(n):
    h = rotate.wht_f64(np.eye(n), axis=0)
    assert np.array_equal(h, scipy_linalg.hadamard(n).astype(np.float64))


def test_wht_matches_sylvester_closed_form():
    n = 128
    h = rotate.wht_f64(np.eye(n), axis=0)
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    closed = np.vectorize(lambda a, b: -1.0 if bin(a & b).count("1") % 2 else 1.0)(i, j)
    assert np.array_equal(h, closed)


@pytest.mark.parametrize("nh,nq,ntok", [(8, 3, 2), (16, 5, 1), (32, 1, 3), (4, 7, 2), (64, 2, 1)])
def test_rotation_matches_dense_kronecker(nh, nq, ntok):
    C = nh * nq
    inp = synth.rotation(C, nh, 40 + nh + nq)
    x = synth.activations(ntok, C, 41 + nh).astype(np.float64)
    dense = np.kron(scipy_linalg.hadamard(nh) / np.sqrt(nh), inp["q"].astype(np.float64))
    s = np.array([-1.0 if (inp["signs"][c // 8] >> (c % 8)) & 1 else 1.0 for c in range(C)])
    want = (dense @ (x * s).T).T
    got = rotate.rotate_f64(x, inp["signs"], inp["q"], nh)
    assert np.allclose(got, want, rtol=0, atol=1e-12 * np.abs(x).sum())


def test_transposed_order_would_fail():
    # Q (x) H differs from H (x) Q: the dense check above separates them
    nh, nq = 8, 3
    inp = synth.rotation(nh * nq, nh, 7)
    a = np.kron(scipy_linalg.hadamard(nh), inp["q"])
    b = np.kron(inp["q"], scipy_linalg.hadamard(nh))
    assert not np.allclose(a, b)


def test_rotation_preserves_norm_and_inverts():
    C, nh = 17408, 1024
    inp = synth.rotation(C, nh, 5)
    x = synth.activations(2, C, 6).astype(np.float64)
    r = rotate.rotate_f64(x, inp["signs"], inp["q"], nh)
    q64 = inp["q"].astype(np.float64)
    qerr = np.abs(q64 @ q64.T - np.eye(17)).max()       # fp32 rounding of an orthogonal matrix
    assert np.allclose(np.linalg.norm(r, axis=1), np.linalg.norm(x, axis=1), rtol=10 * qerr + 1e-12)
    # inverse: x = S (H (x) Q^T) x_rot, with H symmetric and orthonormal
    back = rotate.rotate_f64(r, np.zeros_like(inp["signs"]), q64.T, nh) * rotate.sign_vector(inp["signs"], C)
    assert np.allclose(back, x, rtol=0, atol=1e-5)


def test_exact_orthogonal_q_preserves_norm_exactly():
    # a signed permutation is orthogonal in any precision
    nh, nq = 256, 4
    q = np.zeros((nq, nq))
    for a, (b, sg) in enumerate([(2, 1.0), (0, -1.0), (3, -1.0), (1, 1.0)]):
        q[a, b] = sg
    x = synth.activations(1, nh * nq, 9).astype(np.float64)
    r = rotate.rotate_f64(x, np.full((nh * nq) // 8, 0xA5, dtype=np.uint8), q, nh)
    assert abs(np.linalg.norm(r) - np.linalg.norm(x)) <= 1e-12 * np.linalg.norm(x)


def test_unit_vector_closed_form():
    # S = I, Q = I, x = e_k: x_rot[i*nq + a] = [a == k % nq] * (-1)^popcount(i & (k // nq)) / sqrt(nh)
    nh, nq, k = 64, 3, 50
    x = np.zeros((1, nh * nq))
    x[0, k] = 1.0
    r = rotate.rotate_f64(x, np.zeros((nh * nq + 7) // 8, dtype=np.uint8), np.eye(nq), nh)[0]
    for i in range(nh):
        for a in range(nq):
            want = 0.0 if a != k % nq else (-1.0) ** bin(i & (k // nq)).count("1") / np.sqrt(nh)
            assert r[i * nq + a] == want


def test_abs_bound_is_the_sum_of_term_magnitudes():
    nh, nq = 16, 3
    inp = synth.rotation(nh * nq, nh, 12)
    x = synth.activations(2, nh * nq, 13).astype(np.float64)
    dense = np.abs(np.kron(scipy_linalg.hadamard(nh) / np.sqrt(nh), inp["q"].astype(np.float64)))
    assert np.allclose(rotate.abs_bound(x, inp["signs"], inp["q"], nh), (dense @ np.abs(x).T).T, rtol=1e-12)


def test_default_split_reproduces_the_page_examples():
    facts = json.load(open(GOLDEN))
    for f in facts["splits"]:
        assert rotate.default_split(f["C"]) == (f["nh"], f["nq"])
    assert rotate.default_split(4096) == (2048, 2)
    assert rotate.default_split(12288) == (2048, 6)
