"""The in-launch split-K reduction, on the GPU.

Batch-1 GEMVs (and BPDQ at 2..6 tokens) reduce their per-slice partial sums
inside the launch: every lane adds its slice partial, as a fixed-point
integer with an arrival count, to the 64-bit accumulator word of its row,
and the addition that completes the count writes y and zeroes the word.
These tests check, through the C ABI, that
  - CTAs whose item range spans several slices give results within the
    parity tolerance of the oracle, and more than 255 slices is refused;
  - activations scaled far down or up (the fixed-point scale is set from the
    weights and the fp16 range, not from x) stay within the tolerance;
  - a chain of GEMVs of different formats and shapes sharing one workspace
    on one stream is correct, leaves every accumulator word at zero, and
    gives bit-identical outputs run after run; at 16 and 64 tokens the same
    for the tensor-core path, whose K splits are summed over a thread-block
    cluster in split order (no workspace).
Tolerance: |y - y_ref| <= 2e-3 * sum_c |w x| per output.
"""
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


def _check(y, w64, x, rows=None):
    if rows is not None:
        y = y[:, rows]
    ok = matvec.passes(y, matvec.gemv(w64, x), matvec.abs_bound(w64, x), TOL)
    assert ok.all(), f"{(~ok).sum()} outputs outside the tolerance"


@pytest.mark.parametrize("R,C,seed", [
    (32, 256 * 255, 8000),     # one row block, the most slices a row may have: CTAs span 1..2 slices
    (64, 256 * 200, 8001),     # two row blocks: CTAs span one or two slices
    (96, 256 * 97, 8002),      # ragged: 3 row blocks x 97 slices
])
def test_bpdq_ctas_spanning_many_slices(q2, R, C, seed):
    d = synth.bpdq(R, C, seed)
    w = obpdq.decode_f64(d["plane0"], d["plane1"], d["coef"])
    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=6)
    for ntok in (1, 3, 6):
        x = synth.activations(ntok, C, seed + ntok)
        y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
        _check(y, w, x)
    assert not pk.ws.any().item()


def test_more_than_255_slices_is_refused(q2):
    d = synth.bpdq(32, 256 * 256, 8003)
    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=1)
    x = torch.zeros((1, 256 * 256), dtype=torch.float16, device="cuda")
    y = torch.zeros((1, 32), dtype=torch.float16, device="cuda")
    assert q2.q2_gemv(q2.BPDQ, pk, x, y, 1) == -2


@pytest.mark.parametrize("scale", [1e-4, 3e-3, 40.0])
def test_fixed_point_reduction_at_extreme_activation_scales(q2, scale):
    R, C = 4096, 4096
    d = synth.bpdq(R, C, 8004)
    w = obpdq.decode_f64(d["plane0"], d["plane1"], d["coef"])
    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=16)
    for ntok in (1, 3, 16):
        x = (synth.activations(ntok, C, 8005).astype(np.float64) * scale).astype(np.float16)
        y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
        _check(y, w, x)
    d = synth.leech(512, 5120, 8006)
    x = (synth.activations(1, 5120, 8007).astype(np.float64) * scale).astype(np.float16)
    pk = q2.Packed(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], 5120), ntok_max=1)
    y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
    _check(y, oleech.decode_f64(d["v"], d["scale"], d["tail"]), x)


def test_leech_and_trellis_ctas_spanning_many_slices(q2):
    R, C = 32, 24 * 2600 + 8                       # 244 slices, tail of 8 columns
    d = synth.leech(R, C, 8100)
    x = synth.activations(1, C, 8100)
    pk = q2.Packed(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C), ntok_max=1)
    y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
    _check(y, oleech.decode_f64(d["v"], d["scale"], d["tail"]), x)
    R, C = 64, 256 * 240
    d = synth.trellis(R, C, 8101)
    x = synth.activations(1, C, 8101)
    pk = q2.Packed(q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), ntok_max=1)
    y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
    _check(y, otrellis.decode_f64(d["stream"], d["table"], d["scale"]), x)


def _chain(q2):
    """Matrices of several formats and shapes, in call order."""
    mats = []
    for i, (R, C) in enumerate([(4096, 4096), (6144, 4096), (1024, 12288), (70, 768)]):
        d = synth.bpdq(R, C, 8200 + i)
        mats.append(("bpdq", R, C, d, q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"])))
    d = synth.trellis(2048, 4096, 8210)
    mats.append(("trellis", 2048, 4096, d, q2.q2_pack_trellis(d["stream"], d["table"], d["scale"])))
    d = synth.leech(1000, 5120, 8211)
    mats.append(("leech", 1000, 5120, d, q2.q2_pack_leech(d["v"], d["tail"], d["scale"], 5120)))
    return mats


def _w64(kind, d, rows):
    if kind == "bpdq":
        return obpdq.decode_f64(d["plane0"][rows], d["plane1"][rows], d["coef"][:, rows])
    if kind == "trellis":
        return otrellis.decode_f64(d["stream"][rows], d["table"], d["scale"][rows])
    return oleech.decode_f64(d["v"][rows], d["scale"][rows], d["tail"][rows])


@pytest.mark.parametrize("ntok", [1, 2, 16, 64])
def test_shared_workspace_chain_is_correct_and_repeatable(q2, ntok):
    mats = _chain(q2)
    if ntok > 1:
        # 2..6 tokens share the split-K path in BPDQ only; from 7 the tensor
        # cores sum BPDQ's K split over a cluster (these shapes split K)
        mats = [m for m in mats if m[0] == "bpdq"]
    pks = [q2.Packed(blob, ntok_max=ntok, workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))
           for _, _, _, _, blob in mats]
    ws = torch.zeros(max(16, max(p.workspace_bytes(ntok) for p in pks)), dtype=torch.uint8, device="cuda")
    for p in pks:
        p.set_workspace(ws)
    xs = [torch.from_numpy(synth.activations(ntok, C, 8300 + i)).cuda() for i, (_, _, C, _, _) in enumerate(mats)]
    stream = torch.cuda.Stream()

    def run():
        with torch.cuda.stream(stream):
            ys = [p.gemv(x, stream=stream) for p, x in zip(pks, xs)]
        stream.synchronize()
        return [y.cpu().numpy() for y in ys]

    acc = ws                                # the accumulator words
    plain = run()
    assert not acc.any().item()
    again = [run() for _ in range(3)]
    assert not acc.any().item()
    for h in again:
        for y0, y1 in zip(plain, h):
            assert np.array_equal(y0.view(np.uint16), y1.view(np.uint16))
    for (kind, R, C, d, _), y, x in zip(mats, plain, xs):
        rows = np.unique(np.linspace(0, R - 1, 48).astype(int))
        _check(y, _w64(kind, d, rows), x.cpu().numpy(), rows)


@pytest.mark.parametrize("fmt", ["bpdq", "trellis", "leech", "fp16"])
@pytest.mark.parametrize("slices", [2, 3, 5, 8, 13, 64])
def test_tensor_core_k_split_over_clusters(q2, fmt, slices):
    """K splits of 2..8 CTAs summed over a thread-block cluster, on a ragged
    row count (the last tile's rows past R, and R % 4 != 0, which takes the
    epilogue's scalar stores); every format, 16 tokens."""
    from oracle import fp16 as ofp16
    R, ntok = 201, 16
    C = 256 * slices if fmt != "leech" else 256 * slices + 8       # Leech: C % 24 != 0, a tail
    if fmt == "bpdq":
        d = synth.bpdq(R, C, 8600 + slices)
        blob, w = q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), obpdq.decode_f64(d["plane0"], d["plane1"], d["coef"])
    elif fmt == "trellis":
        d = synth.trellis(R, C, 8610 + slices)
        blob, w = q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), otrellis.decode_f64(d["stream"], d["table"], d["scale"])
    elif fmt == "leech":
        d = synth.leech(R, C, 8620 + slices)
        blob, w = q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C), oleech.decode_f64(d["v"], d["scale"], d["tail"])
    else:
        d = synth.fp16_dense(R, C, 8630 + slices)
        blob, w = q2.q2_pack_fp16(d["w"]), ofp16.decode_f64(d["w"])
    pk = q2.Packed(blob, ntok_max=ntok)
    x = synth.activations(ntok, C, 8640 + slices)
    y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
    _check(y, w, x)
    assert q2.device_errors() == 0
