"""Parity of the CUDA path (through the C ABI) against the oracle.

Every output must satisfy |y - y_ref| <= 2e-3 * sum_c |w[r][c] * x[t][c]|
(fp32 accumulation, fp16 result); decoded weights must equal the oracle's
canonical decode bit for bit.  Inputs come from the seeded generators in
``synth``.
"""
import numpy as np
import pytest

import synth
from oracle import bpdq as obpdq, fp16 as ofp16, leech as oleech, matvec, trellis as otrellis

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


def _run(q2, blob, x, rows=None):
    pk = q2.Packed(blob)
    xd = torch.from_numpy(x).cuda()
    y = pk.gemv(xd)
    torch.cuda.synchronize()
    return pk, y.cpu().numpy()


def _check(y, w64, x, rows=None):
    if rows is not None:
        y = y[:, rows]
    yref = matvec.gemv(w64, x)
    bound = matvec.abs_bound(w64, x)
    ok = matvec.passes(y, yref, bound, TOL)
    rel = matvec.relative_error(y, yref, bound)
    assert ok.all(), f"{(~ok).sum()} outputs fail; worst relative error {rel.max():.3e}"
    return rel.max()


# ------------------------------------------------------------------- BPDQ
@pytest.mark.parametrize("R,C,seed", [(1024, 1024, 0), (70, 768, 1), (32, 256, 2), (1, 512, 3)])
@pytest.mark.parametrize("ntok", [1, 2, 3, 4, 5, 6, 7, 16, 64])
def test_bpdq_parity(q2, R, C, seed, ntok):
    d = synth.bpdq(R, C, seed)
    x = synth.activations(ntok, C, seed)
    _, y = _run(q2, q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), x)
    _check(y, obpdq.decode_f64(d["plane0"], d["plane1"], d["coef"]), x)


@pytest.mark.parametrize("ntok", [16, 48, 64])
def test_bpdq_tensor_path_shapes_and_error_word(q2, ntok):
    # 8B-shaped rows and columns through the tcgen05 path; ragged 128-row tile
    for R, C, seed in [(6144, 4096, 11), (4096, 12288, 12), (160, 512, 13)]:
        d = synth.bpdq(R, C, seed)
        x = synth.activations(ntok, C, seed)
        _, y = _run(q2, q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), x)
        rows = np.unique(np.linspace(0, R - 1, 64).astype(int))
        w = obpdq.decode_f64(d["plane0"][rows], d["plane1"][rows], d["coef"][:, rows])
        _check(y, w, x, rows)
    assert q2.device_errors() == 0


@pytest.mark.parametrize("ntok", [2, 3, 6])
def test_bpdq_multitoken_subset_sum_full_size(q2, ntok):
    # 8B-shaped rows and columns through the 2..6-token CUDA-core path, sampled rows
    for R, C, seed in [(24576, 4096, 21), (4096, 12288, 22)]:
        d = synth.bpdq(R, C, seed)
        x = synth.activations(ntok, C, seed)
        _, y = _run(q2, q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), x)
        rows = _sampled_rows(R, seed=seed)
        w = obpdq.decode_f64(d["plane0"][rows], d["plane1"][rows], d["coef"][:, rows])
        _check(y, w, x, rows)


@pytest.mark.parametrize("ntok", [2, 3, 4, 5, 6])
def test_bpdq_batch_invariant_1_to_6_tokens(q2, ntok):
    # a token's output does not depend on its batch: every token of an
    # ntok-token call (token-pair tables, 2..6 tokens) equals the same token
    # run alone (single-token tables) bit for bit -- same table sums, same
    # accumulation order, integer split-K sums
    for R, C, seed in [(512, 2048, 23), (4096, 4096, 24), (1000, 12288, 25)]:
        d = synth.bpdq(R, C, seed)
        x = synth.activations(ntok, C, seed + ntok)
        pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]))
        yn = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
        for t in range(ntok):
            y1 = pk.gemv(torch.from_numpy(x[t:t + 1].copy()).cuda()).cpu().numpy()
            assert np.array_equal(yn[t].view(np.uint16), y1[0].view(np.uint16)), f"token {t} of {ntok} differs"


def test_bpdq_decode_bit_exact(q2):
    d = synth.bpdq(70, 768, 9)
    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]))
    w = pk.decode().cpu().numpy().view(np.float16).reshape(70, 768)
    assert np.array_equal(w.view(np.uint16), obpdq.decode_fp16(d["plane0"], d["plane1"], d["coef"]).view(np.uint16))


@pytest.mark.parametrize("ntok", [16, 64])
def test_bpdq_tensor_path_one_hot_columns_bit_exact(q2, ntok):
    # x[t] = e_{c_t}: y[t][r] = w[r][c_t] exactly (one nonzero product, fp32
    # accumulation, fp16 result).  The columns c_t cover every column-byte
    # position of a slice and every bit of a byte, in several slices, so a
    # wrong byte or word of the lane un-rotation shows up as a mismatch.
    R, C = 300, 256 * 9
    d = synth.bpdq(R, C, 9100 + ntok)
    w16 = obpdq.decode_fp16(d["plane0"], d["plane1"], d["coef"])
    cols = [(t % 9) * 256 + ((t * 37) % 32) * 8 + (t * 5) % 8 for t in range(ntok)]
    x = np.zeros((ntok, C), dtype=np.float16)
    x[np.arange(ntok), cols] = 1.0
    _, y = _run(q2, q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), x)
    assert np.array_equal(y.view(np.uint16), w16[:, cols].T.view(np.uint16))


def test_bpdq_deterministic_and_repeatable(q2):
    d = synth.bpdq(4096, 4096, 1001)
    x = torch.from_numpy(synth.activations(1, 4096, 1001)).cuda()
    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]))
    ys = [pk.gemv(x).clone() for _ in range(5)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


# ---------------------------------------------------------------- trellis
@pytest.mark.parametrize("R,C,seed", [(100, 1024, 2000), (32, 256, 2001), (257, 512, 2002)])
@pytest.mark.parametrize("ntok", [1, 3, 16, 64])
def test_trellis_parity(q2, R, C, seed, ntok):
    d = synth.trellis(R, C, seed)
    x = synth.activations(ntok, C, seed)
    _, y = _run(q2, q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), x)
    _check(y, otrellis.decode_f64(d["stream"], d["table"], d["scale"]), x)


def test_trellis_decode_bit_exact(q2):
    d = synth.trellis(45, 768, 2010)
    pk = q2.Packed(q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]))
    w = pk.decode().cpu().numpy().view(np.float32).reshape(45, 768)
    assert np.array_equal(w, otrellis.decode_fp32(d["stream"], d["table"], d["scale"]))


# ------------------------------------------------------------------ Leech
def _leech_with_exceptions(R, C, seed):
    d = synth.leech(R, C, seed)
    v = d["v"].copy()
    v[0, 0] = 0
    v[0, 0, 3] = 8                    # (8, 0^23): shell 4, goes to the exception channel
    if R > 5 and v.shape[1] > 7:
        v[5, 7] = 0
        v[5, 7, [1, 2]] = [8, 8]
    d["v"] = v
    return d


LAYOUTS = [0, 1]        # three two's-complement planes + exceptions; four offset-binary planes


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("R,C,seed", [(70, 24 * 40 + 8, 3000), (32, 256, 3001), (100, 5120, 3002), (33, 24, 3003)])
@pytest.mark.parametrize("ntok", [1, 2, 4, 16, 64])
def test_leech_parity(q2, R, C, seed, ntok, layout):
    d = _leech_with_exceptions(R, C, seed)
    x = synth.activations(ntok, C, seed)
    _, y = _run(q2, q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C, layout), x)
    _check(y, oleech.decode_f64(d["v"], d["scale"], d["tail"]), x)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ntok", [1, 2, 16, 64])
def test_leech_width_not_multiple_of_8(q2, ntok, layout):
    # C % 8 != 0: the tensor-core path cannot describe x rows to TMA (row
    # stride not a multiple of 16 bytes) and stages the x tiles and the parity
    # block sums with element loads instead
    R, C = 70, 24 * 20 + 12
    d = _leech_with_exceptions(R, C, 3100 + ntok)
    x = synth.activations(ntok, C, 3101)
    _, y = _run(q2, q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C, layout), x)
    _check(y, oleech.decode_f64(d["v"], d["scale"], d["tail"]), x)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ntok", [1, 16])
def test_leech_one_hot_columns_bit_exact(q2, layout, ntok):
    """A unit vector x = e_c selects one weight per row: y[r] = fp16(v[r][c] x
    (scale_r x 1/sqrt(8))) in fp32, exactly what both kernels compute for it
    (the subset sums at one token, the tensor-core decode at 16), for columns
    that include every planted v = +8 and some of its -8 neighbours."""
    R, C = 70, 24 * 40 + 8
    d = _leech_with_exceptions(R, C, 3020)
    pk = q2.Packed(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C, layout), ntok_max=ntok)
    cols = [3, 7 * 24 + 1, 7 * 24 + 2, 0, 5, 100, 250, 256, 511, 700, 24 * 40 - 1] + list(range(300, 305))
    vf = d["v"].reshape(R, -1).astype(np.float32)
    post = np.float32(q2.INV_SQRT8_F32)
    sc = d["scale"].astype(np.float32)
    for k in range(0, len(cols), ntok):
        batch = cols[k:k + ntok]
        x = np.zeros((ntok, C), dtype=np.float16)
        for t, c in enumerate(batch):
            x[t, c] = 1.0
        y = pk.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
        for t, c in enumerate(batch):
            want = (vf[:, c] * (sc * post)).astype(np.float16)
            assert np.array_equal(y[t].view(np.uint16), want.view(np.uint16)), f"column {c}"


@pytest.mark.parametrize("layout", LAYOUTS)
def test_leech_decode_bit_exact(q2, layout):
    R, C = 70, 24 * 40 + 8
    d = _leech_with_exceptions(R, C, 3010)
    pk = q2.Packed(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C, layout))
    out = pk.decode().cpu().numpy()
    body = R * 40 * 24
    v = out[:body].view(np.int8).reshape(R, 40, 24)
    assert np.array_equal(v, d["v"])
    start = (body + 15) // 16 * 16
    tail = out[start:start + R * 8 * 2].view(np.float16).reshape(R, 8)
    assert np.array_equal(tail.view(np.uint16), d["tail"].view(np.uint16))


# ---------------------------------------------------------------- fp16
# One token on CUDA cores, 2..64 through the tensor-core kernel with plain
# row loads: ragged rows (R % 128 != 0), a partial last 256-column slice
# (C % 256 != 0), a single short row, and a K split reduced by the second
# launch (17408 columns).
@pytest.mark.parametrize("R,C", [(300, 1032), (1, 8), (129, 4104)])
@pytest.mark.parametrize("ntok", [1, 2, 3, 7, 16, 33, 64])
def test_fp16_parity(q2, R, C, ntok):
    d = synth.fp16_dense(R, C, 4000 + R)
    x = synth.activations(ntok, C, 4000)
    _, y = _run(q2, q2.q2_pack_fp16(d["w"]), x)
    _check(y, ofp16.decode_f64(d["w"]), x)


@pytest.mark.parametrize("ntok", [2, 16, 64])
def test_fp16_tensor_path_full_size(q2, ntok):
    R, C = 5120, 17408
    d = synth.fp16_dense(R, C, 4100)
    x = synth.activations(ntok, C, 4101)
    _, y = _run(q2, q2.q2_pack_fp16(d["w"]), x)
    rows = _sampled_rows(R, seed=4102)
    _check(y, ofp16.decode_f64(d["w"][rows]), x, rows)
    assert q2.device_errors() == 0


def test_fp16_tensor_path_one_hot_bit_exact(q2):
    # x = e_c per token selects one weight per row: y[t][r] = w[r][c_t]
    # exactly (one fp32 product by 1.0, rounded back to fp16), which pins the
    # order in which the rows reach tensor memory column by column
    R, C = 200, 776
    d = synth.fp16_dense(R, C, 4200)
    cols = np.array([0, 1, 7, 8, 63, 64, 255, 256, 511, 512, 700, 767, 768, 775] + list(range(100, 150)))   # 64 tokens
    x = np.zeros((len(cols), C), dtype=np.float16)
    x[np.arange(len(cols)), cols] = 1.0
    _, y = _run(q2, q2.q2_pack_fp16(d["w"]), x)
    assert np.array_equal(y.view(np.uint16), d["w"][:, cols].T.view(np.uint16))


def test_noweights_control_runs(q2):
    pk = q2.Packed(q2.q2_pack_noweights(1024, 1024))
    x = torch.from_numpy(synth.activations(1, 1024, 5)).cuda()
    y1 = pk.gemv(x).clone()
    y2 = pk.gemv(x)
    torch.cuda.synchronize()
    assert torch.isfinite(y1.float()).all() and torch.equal(y1, y2)


# ------------------------------------------------------- full-size shapes
def _sampled_rows(R, n=96, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(R, size=min(n, R), replace=False))
    rows[0], rows[-1] = 0, R - 1
    return np.unique(rows)


@pytest.mark.parametrize("R,C", [(6144, 4096), (4096, 4096), (24576, 4096), (4096, 12288)])
def test_bpdq_full_size_8b_layers(q2, R, C):
    seed = 1000 + R + C
    d = synth.bpdq(R, C, seed)
    x = synth.activations(1, C, seed)
    _, y = _run(q2, q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), x)
    rows = _sampled_rows(R)
    w = obpdq.decode_f64(d["plane0"][rows], d["plane1"][rows], d["coef"][:, rows])
    _check(y, w, x, rows)


@pytest.mark.parametrize("R,C", [(12288, 4096), (4096, 12288)])
def test_trellis_full_size(q2, R, C):
    d = synth.trellis(R, C, 2000 + (R > C))
    x = synth.activations(1, C, 2000 + (R > C))
    _, y = _run(q2, q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), x)
    rows = _sampled_rows(R)
    _check(y, otrellis.decode_f64(d["stream"][rows], d["table"], d["scale"][rows]), x, rows)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("R,C", [(17408, 5120), (5120, 17408)])
def test_leech_full_size(q2, R, C, layout):
    d = synth.leech(R, C, 3000 + (R > C))
    x = synth.activations(1, C, 3000 + (R > C))
    _, y = _run(q2, q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C, layout), x)
    rows = _sampled_rows(R)
    _check(y, oleech.decode_f64(d["v"][rows], d["scale"][rows], d["tail"][rows]), x, rows)
