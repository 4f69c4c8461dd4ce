"""The row limit on the GPU: R = 524288 (the most rows a handle may have)
runs on every format and path, and one row more is refused.

At the limit the CUDA-core kernels cover 16384 row blocks in one slice and
the tensor-core kernel 4096 tiles; the accumulator workspace holds the
largest word count it is sized for.  Outputs are compared with the oracle on
sampled rows, always including the first and the last.
Tolerance: |y - y_ref| <= 2e-3 * sum_c |w x|.
"""
import numpy as np
import pytest

import synth
from oracle import bpdq as obpdq, fp16 as ofp16, leech as oleech, matvec, trellis as otrellis

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

R_MAX = 524288
ESHAPE = -2


@pytest.fixture(scope="module")
def q2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dequant_gemv_q2_gb300 as m
    m.load(build_if_missing=True)
    return m


def _rows(R, seed):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(R, size=128, replace=False))
    rows[0], rows[-1] = 0, R - 1
    return np.unique(rows)


def _case(q2, fmt, R, seed):
    """(blob, C, oracle decode of the given rows)."""
    if fmt == "bpdq":
        C = 256
        d = synth.bpdq(R, C, seed)
        return (q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), C,
                lambda r: obpdq.decode_f64(d["plane0"][r], d["plane1"][r], d["coef"][:, r]))
    if fmt == "trellis":
        C = 256
        d = synth.trellis(R, C, seed)
        return (q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), C,
                lambda r: otrellis.decode_f64(d["stream"][r], d["table"], d["scale"][r]))
    if fmt == "leech":
        C = 48
        d = synth.leech(R, C, seed)
        return (q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C), C,
                lambda r: oleech.decode_f64(d["v"][r], d["scale"][r], d["tail"][r]))
    C = 64
    d = synth.fp16_dense(R, C, seed)
    return q2.q2_pack_fp16(d["w"]), C, lambda r: ofp16.decode_f64(d["w"][r])


@pytest.mark.parametrize("fmt,ntoks", [("bpdq", (1, 3, 16)), ("trellis", (1, 16)), ("leech", (1, 2, 16)),
                                       ("fp16", (1, 16))])
def test_maximum_rows(q2, fmt, ntoks):
    seed = 9100 + len(fmt)
    blob, C, decode = _case(q2, fmt, R_MAX, seed)
    rows = _rows(R_MAX, seed)
    w = decode(rows)
    pk = q2.Packed(blob, ntok_max=max(ntoks))
    for ntok in ntoks:
        x = synth.activations(ntok, C, seed + ntok)
        y = pk.gemv(torch.from_numpy(x).cuda())
        torch.cuda.synchronize()
        assert q2.device_errors() == 0
        yh = y.cpu().numpy()
        assert np.isfinite(yh.astype(np.float32)).all(), f"{fmt} at {ntok} tokens: an output was not written"
        ys = yh[:, rows].astype(np.float64)
        ok = matvec.passes(ys, matvec.gemv(w, x), matvec.abs_bound(w, x), 2e-3)
        assert ok.all(), f"{fmt} at {ntok} tokens: {(~ok).sum()} sampled outputs outside the tolerance"


def test_one_row_past_the_limit_is_refused(q2):
    d = synth.bpdq(R_MAX + 1, 256, 9200)
    blob = q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"])
    with pytest.raises(q2.Q2Error) as e:
        pk = q2.Packed(blob)
        pk.gemv(torch.zeros((1, 256), dtype=torch.float16, device="cuda"))
        torch.cuda.synchronize()
    assert e.value.status == ESHAPE
