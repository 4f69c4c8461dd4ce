"""The tensor-core kernel's bounded waits, made to run out on purpose.

Every wait in the tensor-core kernel is bounded.  A test hook
(q2_debug_wait_limit) shortens only the helper warp's stage waits (a
slice's decoded weights and x tile ready) to a single poll, so they give up
before the decoders can finish; the roles then stop waiting on each other,
the CTA waits with the full bound for its x copies and MMAs still in flight,
puts NaN in place of its partial sums, still meets its cluster at both
barriers (a K split's CTAs sum their partials together), frees its tensor
memory and exits.  Nothing faults and nothing hangs: the host reads a
nonzero error word, the rows of the tiles that gave up are NaN, the
workspace is untouched, and the next call with the normal bound is correct
again.  Tolerance for the normal calls: |y - y_ref| <= 2e-3 * sum_c |w x|.
"""
import numpy as np
import pytest

import synth
from oracle import bpdq as obpdq, matvec, trellis as otrellis

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dequant_gemv_q2_gb300 as m
    m.load(build_if_missing=True)
    m.debug_wait_limit(0)
    m.device_errors()                          # start from a clear error word
    yield m
    m.debug_wait_limit(0)


def _passes(y, w, x):
    return matvec.passes(y, matvec.gemv(w, x), matvec.abs_bound(w, x), 2e-3).all()


def test_stage_wait_timeout_reports_error_and_leaves_workspace_clean(q2):
    # BPDQ 1024 x 4096 at 16 tokens: 8 row tiles, K split over clusters
    R, C, ntok = 1024, 4096, 16
    d = synth.bpdq(R, C, 9600)
    w = obpdq.decode_f64(d["plane0"], d["plane1"], d["coef"])
    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=ntok)
    x = synth.activations(ntok, C, 9601)
    xd = torch.from_numpy(x).cuda()
    q2.debug_wait_limit(1)
    try:
        y = pk.gemv(xd).cpu().numpy()
    finally:
        q2.debug_wait_limit(0)
    err = q2.device_errors()
    assert err != 0
    assert np.isnan(y.astype(np.float32)).any()          # rows of the tiles that gave up
    if pk.ws is not None:
        assert not pk.ws.any().item()                    # the accumulator words are untouched
    # the next call with the normal bound is correct and reports nothing
    y2 = pk.gemv(xd).cpu().numpy()
    assert q2.device_errors() == 0
    assert _passes(y2, w, x)


def test_stage_wait_timeout_with_a_row_epilogue(q2):
    # trellis at 16 tokens: the cluster's sum is scaled per row before y
    R, C, ntok = 512, 2048, 16
    d = synth.trellis(R, C, 9610)
    w = otrellis.decode_f64(d["stream"], d["table"], d["scale"])
    pk = q2.Packed(q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), ntok_max=ntok)
    x = synth.activations(ntok, C, 9611)
    xd = torch.from_numpy(x).cuda()
    q2.debug_wait_limit(1)
    try:
        pk.gemv(xd)
        torch.cuda.synchronize()
    finally:
        q2.debug_wait_limit(0)
    assert q2.device_errors() != 0
    y2 = pk.gemv(xd).cpu().numpy()
    assert q2.device_errors() == 0
    assert _passes(y2, w, x)


def test_wait_limit_rejects_negative(q2):
    L = q2.load()
    assert L.q2_debug_wait_limit(-1) == -1
