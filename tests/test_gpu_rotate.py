"""Parity of the activation rotation x_rot = (H (x) Q)(S x) (``q2_rotate``,
"Qwen3.8-27B on a 12 GB card", section "What the kernel does per token")
against the f64 oracle ``oracle.rotate``.

The kernel computes in fp32 and rounds once to fp16, so each output must
satisfy |x_rot - ref| <= 2^-11 |ref| + 2^-24 + k * bound, where bound is the
sum of the magnitudes of the output's terms and k = (nq + log2(nh) + 2) *
2^-23 covers the fp32 multiply-adds of Q and the butterfly stages.
"""
import math

import numpy as np
import pytest

import synth
from oracle import rotate as orot

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dequant_gemv_q2_gb300 as m
    m.load(build_if_missing=True)
    return m


def _check(got, x, inp, nh):
    ref = orot.rotate_f64(x, inp["signs"], inp["q"], nh)
    bound = orot.abs_bound(x, inp["signs"], inp["q"], nh)
    k = (inp["nq"] + math.log2(nh) + 2) * 2.0 ** -23
    err = np.abs(got.astype(np.float64) - ref)
    tol = 2.0 ** -11 * np.abs(ref) + 2.0 ** -24 + k * bound
    assert (err <= tol).all(), f"{(err > tol).sum()} outputs outside the bound; worst {(err / tol).max():.2f}x"


def _run(q2, inp, x, nh, q=True):
    rot = q2.Rotation(inp["signs"], inp["q"] if q else None, nh, x.shape[1])
    return rot.apply(torch.from_numpy(x).cuda()).cpu().numpy()


@pytest.mark.parametrize("C", [17408, 6144, 5120, 4096, 12288, 1024])
@pytest.mark.parametrize("ntok", [1, 3, 64])
def test_rotation_parity_page_widths(q2, C, ntok):
    nh, nq = q2.q2_rotate_split(C)
    inp = synth.rotation(C, nh, 500 + C % 997)
    x = synth.activations(ntok, C, 501 + ntok)
    _check(_run(q2, inp, x, nh), x, inp, nh)


@pytest.mark.parametrize("C,nh", [(24, 8), (96, 32), (2, 2), (32, 1), (31 * 64, 64), (7 * 128, 128), (49152, 2048)])
def test_rotation_parity_other_splits(q2, C, nh):
    # every pass width 1..5, nq from 1 to 32, the largest C
    inp = synth.rotation(C, nh, 600 + C)
    x = synth.activations(2, C, 601)
    _check(_run(q2, inp, x, nh), x, inp, nh)


def test_rotation_without_q_is_signs_then_hadamard(q2):
    C, nh = 4096, 4096
    inp = synth.rotation(C, nh, 700)                    # nq = 1: q may be omitted (Q = [1])
    x = synth.activations(4, C, 701)
    got = _run(q2, inp, x, nh, q=False)
    _check(got, x, dict(inp, q=np.ones((1, 1), dtype=np.float32)), nh)


def test_rotation_of_a_unit_vector_is_exact(q2):
    # S = +1, Q = I: e_k maps to +-1/sqrt(nh) on run position k % nq, exactly representable in fp16
    nh, nq, k = 1024, 4, 1234
    C = nh * nq
    x = np.zeros((1, C), dtype=np.float16)
    x[0, k] = 1.0
    inp = {"signs": np.zeros(C // 8, dtype=np.uint8), "q": np.eye(nq, dtype=np.float32), "nq": nq}
    got = _run(q2, inp, x, nh).astype(np.float64)[0]
    want = orot.rotate_f64(x, inp["signs"], inp["q"], nh)[0]
    assert np.array_equal(got, want)


def test_rotation_refuses_bad_shapes(q2):
    d = torch.zeros(64, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 4096), dtype=torch.float16, device="cuda")
    y = torch.zeros_like(x)
    q = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    assert q2.q2_rotate(x, y, 1, 4096, 1000, d, q) == -2           # nh not a power of two
    assert q2.q2_rotate(x, y, 1, 4096, 64, d, q) == -2             # nq = 64 > 32
    assert q2.q2_rotate(x, y, 1, 4095, 1024, d, q) == -2           # C not a multiple of nh
    assert q2.q2_rotate(x, y, 1, 4096, 1024, d, None) == -1        # nq = 4 needs Q
    assert q2.q2_rotate(x, x, 1, 4096, 4096, d, None) == -1        # in place is refused
    assert q2.q2_rotate(x, y, 0, 4096, 4096, d, None) == -5        # ntok outside 1..64
    torch.cuda.synchronize()
