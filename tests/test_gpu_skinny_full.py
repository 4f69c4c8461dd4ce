"""Parity of the skinny path at the full sizes of the benchmarks: the
Qwen3-14B stack's shapes (qkv 7168x5120, gate_up 34816x5120, down
5120x17408), trellis 12288x4096 / 4096x12288 and Leech 17408x5120, at 3, 16 and 64
tokens, in the launch configurations the sweep times (tensor-core path with
its K split and reduction; BPDQ at 3 tokens as a token pair plus a single
token).  The oracle computes sampled rows only.  Tolerance as everywhere:
|y - y_ref| <= 2e-3 * sum_c |w x| per output."""
import numpy as np
import pytest

import synth
from oracle import bpdq as obpdq, leech as oleech, matvec, trellis as otrellis

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def q2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dequant_gemv_q2_gb300 as m
    m.load(build_if_missing=True)
    return m


def _rows(R, n=48, seed=0):
    rng = np.random.default_rng(seed + R)
    return np.unique(np.concatenate([[0, R - 1], rng.integers(0, R, size=n)]))


def _check(y, w, x, rows):
    y = y[:, rows]
    ok = matvec.passes(y, matvec.gemv(w, x), matvec.abs_bound(w, x), TOL)
    assert ok.all(), f"{(~ok).sum()} sampled outputs outside the tolerance"


@pytest.mark.parametrize("R,C", [(7168, 5120), (34816, 5120), (5120, 17408)])
@pytest.mark.parametrize("ntok", [3, 16, 64])
def test_bpdq_14b_shapes(q2, R, C, ntok):
    d = synth.bpdq(R, C, 7000 + R % 997)
    x = synth.activations(ntok, C, 7001)
    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=ntok)
    y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
    rows = _rows(R)
    _check(y, obpdq.decode_f64(d["plane0"][rows], d["plane1"][rows], d["coef"][:, rows]), x, rows)
    assert q2.device_errors() == 0


@pytest.mark.parametrize("R,C", [(12288, 4096), (4096, 12288)])
@pytest.mark.parametrize("ntok", [16, 64])
def test_trellis_full_size_skinny(q2, R, C, ntok):
    d = synth.trellis(R, C, 7100 + (R > C))
    x = synth.activations(ntok, C, 7101)
    pk = q2.Packed(q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), ntok_max=ntok)
    y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
    rows = _rows(R)
    _check(y, otrellis.decode_f64(d["stream"][rows], d["table"], d["scale"][rows]), x, rows)
    assert q2.device_errors() == 0


def test_leech_full_size_skinny(q2):
    # one 17408 x 5120 matrix (its generation is the slow part) at 2 tokens
    # (two single-token launches) and 64 tokens (tensor cores)
    R, C = 17408, 5120
    d = synth.leech(R, C, 7200)
    pk = q2.Packed(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C), ntok_max=64)
    rows = _rows(R)
    w = oleech.decode_f64(d["v"][rows], d["scale"][rows], d["tail"][rows])
    for ntok in (2, 64):
        x = synth.activations(ntok, C, 7201 + ntok)
        y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
        _check(y, w, x, rows)
    assert q2.device_errors() == 0
