"""Non-finite activations on the GPU.

In IEEE arithmetic one inf or NaN in a token's x makes every output of that
token non-finite (every row has a weight in that column, and 0 x inf is
NaN); the oracle (f64 numpy) shows it.  The fixed-point split-K sums of
the CUDA-core paths cannot carry infs or NaNs, so those kernels flag them
in the accumulator word; the tensor-core path sums fp32 partials (in a
cluster's shared memory), which carry them.  These tests put an inf in one
token and a NaN in another, at 1 token (every format), 3 tokens (BPDQ
token pairs) and 16 tokens (the tensor-core path, with and without a K
split), and check that exactly the affected tokens' outputs are non-finite
while the other tokens still match the oracle.
Tolerance for the finite tokens: |y - y_ref| <= 2e-3 * sum_c |w x|.
"""
import numpy as np
import pytest

import synth
from oracle import bpdq as obpdq, leech as oleech, matvec, trellis as otrellis

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dequant_gemv_q2_gb300 as m
    m.load(build_if_missing=True)
    return m


def _bpdq(q2, R, C, seed, ntok):
    d = synth.bpdq(R, C, seed)
    return q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=ntok), \
        obpdq.decode_f64(d["plane0"], d["plane1"], d["coef"])


def _trellis(q2, R, C, seed, ntok):
    d = synth.trellis(R, C, seed)
    return q2.Packed(q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), ntok_max=ntok), \
        otrellis.decode_f64(d["stream"], d["table"], d["scale"])


def _leech(q2, R, C, seed, ntok):
    d = synth.leech(R, C, seed)
    return q2.Packed(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C), ntok_max=ntok), \
        oleech.decode_f64(d["v"], d["scale"], d["tail"])


CASES = [
    ("bpdq", 1024, 4096, 1),     # single-token kernel, 16 slices
    ("bpdq", 2048, 12288, 1),    # 48 slices
    ("bpdq", 512, 2048, 3),      # token pairs + single token
    ("bpdq", 256, 2048, 16),     # tensor cores, K split over a cluster
    ("bpdq", 256, 4096, 16),     # tensor cores, a wider K split
    ("trellis", 512, 2048, 1),
    ("trellis", 256, 2048, 16),
    ("leech", 544, 1040, 1),
    ("leech", 256, 1040, 16),
]


@pytest.mark.parametrize("fmt,R,C,ntok", CASES)
def test_inf_and_nan_in_x_make_exactly_those_tokens_non_finite(q2, fmt, R, C, ntok):
    make = {"bpdq": _bpdq, "trellis": _trellis, "leech": _leech}[fmt]
    pk, w = make(q2, R, C, 9500 + R + C, ntok)
    x = synth.activations(ntok, C, 9501).astype(np.float16)
    bad = {0: (5, np.inf)} if ntok == 1 else {0: (5, np.inf), ntok - 1: (C - 1, np.nan)}
    for t, (c, v) in bad.items():
        x[t, c] = v
    y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy().astype(np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        yref = matvec.gemv(w, x)
        bound = matvec.abs_bound(w, x)
    for t in range(ntok):
        if t in bad:
            assert not np.isfinite(yref[t]).any()                      # the oracle: every output non-finite
            assert not np.isfinite(y[t]).any(), f"token {t}: {np.isfinite(y[t]).sum()} finite outputs"
        else:
            ok = matvec.passes(y[t:t + 1], yref[t:t + 1], bound[t:t + 1], 2e-3)
            assert ok.all(), f"token {t}: {(~ok).sum()} outputs outside the tolerance"
    if pk.ws is not None:
        acc_words = ntok * ((R + 31) // 32 * 32) * 8
        assert not pk.ws[:acc_words].any().item()                      # the accumulator words are back at zero
    # the next call on clean input is exact again
    x2 = synth.activations(ntok, C, 9502)
    y2 = pk.gemv(torch.from_numpy(x2).cuda()).cpu().numpy()
    ok = matvec.passes(y2, matvec.gemv(w, x2), matvec.abs_bound(w, x2), 2e-3)
    assert ok.all()
