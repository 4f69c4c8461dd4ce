"""Guard regions around every buffer a GEMV touches, on the GPU.

x sits between NaN guards: a read past either end of x (or of one token's
row) would make outputs NaN, so every output must be finite and within the
oracle's tolerance.  y and the workspace sit between sentinel guards that
must be unchanged after the call (a write past either end, or into another
token's row, would change them), and the workspace's accumulator words must
be back at zero.  Shapes are ragged (R not a multiple of 32 or 128, C with a
partial last slice where the format allows) and cover every path: one token
per format, BPDQ token pairs, Leech at 2 tokens, the tensor cores with and
without a K split, the fp16 control, the no-weights control, and the
activation rotation.
Tolerance: |y - y_ref| <= 2e-3 * sum_c |w x|.
"""
import numpy as np
import pytest

import synth
from oracle import bpdq as obpdq, fp16 as ofp16, leech as oleech, matvec, trellis as otrellis

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

G = 512                      # guard elements on each side (1 KiB of fp16: keeps 16-byte alignment)
SENT = 0x5A5A                # fp16 sentinel bits of the y guards
WS_SENT = 0xA5               # byte sentinel of the workspace guards


@pytest.fixture(scope="module")
def q2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dequant_gemv_q2_gb300 as m
    m.load(build_if_missing=True)
    return m


def _packed(q2, fmt, R, C, seed):
    if fmt == "bpdq":
        d = synth.bpdq(R, C, seed)
        return q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), obpdq.decode_f64(d["plane0"], d["plane1"], d["coef"])
    if fmt == "trellis":
        d = synth.trellis(R, C, seed)
        return q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), otrellis.decode_f64(d["stream"], d["table"], d["scale"])
    if fmt == "leech":
        d = synth.leech(R, C, seed)
        return q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C), oleech.decode_f64(d["v"], d["scale"], d["tail"])
    d = synth.fp16_dense(R, C, seed)
    return q2.q2_pack_fp16(d["w"]), ofp16.decode_f64(d["w"])


CASES = [
    ("bpdq", 1, 201, 1280), ("bpdq", 3, 201, 1280), ("bpdq", 16, 201, 1280), ("bpdq", 64, 330, 4096),
    ("trellis", 1, 201, 1280), ("trellis", 16, 201, 2048), ("trellis", 64, 130, 1024),
    ("leech", 1, 201, 1040), ("leech", 2, 200, 1040), ("leech", 16, 201, 1048), ("leech", 64, 130, 2056),
    ("fp16", 1, 201, 1032), ("fp16", 16, 201, 1032), ("fp16", 64, 130, 2056),
]


@pytest.mark.parametrize("fmt,ntok,R,C", CASES)
def test_gemv_stays_inside_its_buffers(q2, fmt, ntok, R, C):
    blob, w = _packed(q2, fmt, R, C, 7700 + R + C + ntok)
    pk = q2.Packed(blob, ntok_max=ntok)
    x = synth.activations(ntok, C, 7701)
    # x between NaN guards
    xbuf = torch.full((G + ntok * C + G,), float("nan"), dtype=torch.float16, device="cuda")
    xbuf[G:G + ntok * C].copy_(torch.from_numpy(x.reshape(-1)).cuda())
    xd = xbuf[G:G + ntok * C].view(ntok, C)
    # y between sentinel guards
    ybuf = torch.full((G + ntok * R + G,), 0, dtype=torch.int16, device="cuda")
    ybuf.fill_(SENT)
    yd = ybuf[G:G + ntok * R].view(torch.float16).view(ntok, R)
    # the workspace between sentinel guards (its own region zero, as required)
    need = pk.workspace_bytes(ntok)
    if need:
        wbuf = torch.full((256 + need + 256,), WS_SENT, dtype=torch.uint8, device="cuda")
        wbuf[256:256 + need].zero_()
        pk.set_workspace(wbuf[256:256 + need])
    pk.gemv(xd, yd)
    torch.cuda.synchronize()
    assert q2.device_errors() == 0
    yb = ybuf.cpu().numpy()
    assert (yb[:G] == SENT).all() and (yb[G + ntok * R:] == SENT).all(), "a write landed outside y"
    y = yd.cpu().numpy().astype(np.float64)
    assert np.isfinite(y).all(), "an output read past x (NaN guard) or was not written"
    ok = matvec.passes(y, matvec.gemv(w, x), matvec.abs_bound(w, x), 2e-3)
    assert ok.all(), f"{(~ok).sum()} outputs outside the tolerance"
    if need:
        wb = wbuf.cpu().numpy()
        assert (wb[:256] == WS_SENT).all() and (wb[256 + need:] == WS_SENT).all(), "a write landed outside the workspace"
        assert not wb[256:256 + need].any(), "accumulator words not back at zero"


def test_noweights_control_stays_inside_y(q2):
    R, C = 201, 1280
    pk = q2.Packed(q2.q2_pack_noweights(R, C), ntok_max=1)
    xbuf = torch.zeros((G + C + G,), dtype=torch.float16, device="cuda")
    ybuf = torch.full((G + R + G,), SENT, dtype=torch.int16, device="cuda")
    pk.gemv(xbuf[G:G + C].view(1, C), ybuf[G:G + R].view(torch.float16).view(1, R))
    torch.cuda.synchronize()
    yb = ybuf.cpu().numpy()
    assert (yb[:G] == SENT).all() and (yb[G + R:] == SENT).all()


@pytest.mark.parametrize("C,ntok", [(5120, 1), (17408, 3), (4096, 64)])
def test_rotation_stays_inside_its_buffers(q2, C, ntok):
    nh, nq = q2.q2_rotate_split(C)
    r = synth.rotation(C, nh, seed=7800 + C)
    rot = q2.Rotation(r["signs"], r["q"], nh, C)
    x = synth.activations(ntok, C, 7801)
    xbuf = torch.full((G + ntok * C + G,), float("nan"), dtype=torch.float16, device="cuda")
    xbuf[G:G + ntok * C].copy_(torch.from_numpy(x.reshape(-1)).cuda())
    obuf = torch.full((G + ntok * C + G,), SENT, dtype=torch.int16, device="cuda")
    out = obuf[G:G + ntok * C].view(torch.float16).view(ntok, C)
    rot.apply(xbuf[G:G + ntok * C].view(ntok, C), out)
    torch.cuda.synchronize()
    ob = obuf.cpu().numpy()
    assert (ob[:G] == SENT).all() and (ob[G + ntok * C:] == SENT).all(), "a write landed outside x_rot"
    assert np.isfinite(out.cpu().numpy().astype(np.float32)).all(), "a read past x (NaN guard)"
