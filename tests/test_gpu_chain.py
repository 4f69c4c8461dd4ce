"""q2_gemv_chain on the GPU: a decode step's GEMVs launched in order, each
launch prefetching the weights of the next ones into L2.

The prefetch only moves bytes into L2, so the chain must give exactly the
outputs of the same q2_gemv calls made one by one, bit for bit, at every
lookahead; the shared workspace's accumulator words must be zero after it;
and a chain whose y feeds the next GEMV's x (a true dependency) must match
the oracle run in the same order.
Tolerance for the oracle comparison: |y - y_ref| <= 2e-3 * sum_c |w x|.
"""
import numpy as np
import pytest

import synth
from oracle import bpdq as obpdq, matvec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dequant_gemv_q2_gb300 as m
    m.load(build_if_missing=True)
    return m


def _mats(q2, ntok):
    """Six matrices of three formats and several shapes (small enough for the test)."""
    out = []
    for i, (R, C) in enumerate([(1024, 1024), (3072, 2048), (2048, 3072)]):
        d = synth.bpdq(R, C, 9100 + i)
        out.append(q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=ntok))
    if ntok == 1:
        d = synth.trellis(1024, 2048, 9110)
        out.append(q2.Packed(q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), ntok_max=1))
        d = synth.leech(544, 1040, 9111)
        out.append(q2.Packed(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], 1040), ntok_max=1))
    out.append(q2.Packed(q2.q2_pack_noweights(2048, 1024), ntok_max=1) if ntok == 1 else out[0])
    return out


@pytest.mark.parametrize("ntok", [1, 2, 5])
def test_chain_is_bit_identical_to_separate_calls(q2, ntok):
    pks = _mats(q2, ntok)
    need = max(p.workspace_bytes(ntok) for p in pks)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for p in pks:
        p.set_workspace(ws)
    xs = [torch.from_numpy(synth.activations(ntok, p.C, 9200 + i)).cuda() for i, p in enumerate(pks)]
    ref = [p.gemv(x) for p, x in zip(pks, xs)]
    torch.cuda.synchronize()
    for la in range(0, 5):
        ys = [torch.full((ntok, p.R), float("nan"), dtype=torch.float16, device="cuda") for p in pks]
        q2.Chain(list(zip(pks, xs, ys)), ntok, la).run()
        torch.cuda.synchronize()
        for r, y in zip(ref, ys):
            assert torch.equal(r.view(torch.int16), y.view(torch.int16)), f"lookahead {la}"
        assert not ws.any().item()


def test_chain_with_true_dependency_matches_oracle(q2):
    """y of each GEMV is the next GEMV's x (square BPDQ matrices), run twice:
    the second run, after the words were reset, gives the same bits."""
    C = 2048
    ds = [synth.bpdq(C, C, 9300 + i) for i in range(4)]
    pks = [q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=1) for d in ds]
    ws = torch.zeros(max(p.workspace_bytes(1) for p in pks), dtype=torch.uint8, device="cuda")
    for p in pks:
        p.set_workspace(ws)
    x0 = synth.activations(1, C, 9310)
    bufs = [torch.from_numpy(x0).cuda()] + [torch.empty((1, C), dtype=torch.float16, device="cuda") for _ in pks]
    chain = q2.Chain([(p, bufs[i], bufs[i + 1]) for i, p in enumerate(pks)], 1, 2)
    chain.run()
    torch.cuda.synchronize()
    first = [b.clone() for b in bufs[1:]]
    # the oracle in the same order, from the GPU's own fp16 inputs at each step
    x = x0
    for i, d in enumerate(ds):
        w = obpdq.decode_f64(d["plane0"], d["plane1"], d["coef"])
        y = first[i].cpu().numpy()
        ok = matvec.passes(y, matvec.gemv(w, x), matvec.abs_bound(w, x), 2e-3)
        assert ok.all(), f"GEMV {i}: {(~ok).sum()} outputs outside the tolerance"
        x = y
    chain.run()
    torch.cuda.synchronize()
    for a, b in zip(first, bufs[1:]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not ws.any().item()


def test_chain_refuses_bad_arguments_before_launching(q2):
    d = synth.bpdq(256, 256, 9400)
    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=1)
    x = torch.from_numpy(synth.activations(1, 256, 9401)).cuda()
    y = torch.full((1, 256), 7.0, dtype=torch.float16, device="cuda")
    with pytest.raises(q2.Q2Error):
        q2.Chain([(pk, x, y)], 1, 5).run()                 # lookahead above 4
    ch = q2.Chain([(pk, x, y), (pk, x, y)], 1, 1)
    ch._fmt[1] = q2.TRELLIS                                 # wrong format for the second handle
    with pytest.raises(q2.Q2Error):
        ch.run()
    torch.cuda.synchronize()
    assert (y == 7.0).all().item()                          # nothing was launched


@pytest.mark.parametrize("fmt", ["bpdq", "trellis", "leech", "fp16"])
@pytest.mark.parametrize("ntok", [16, 64])
def test_tensor_core_chain_with_true_dependency_matches_oracle(q2, fmt, ntok):
    """The tensor-core kernel waits for the previous kernel only where it reads
    x and before it writes y (its weights are decoded before the wait): a chain
    whose y is the next GEMV's x, launched back to back, must match the oracle
    run in the same order from the GPU's own fp16 inputs."""
    from oracle import fp16 as ofp16, leech as oleech, trellis as otrellis
    C = 2048 if fmt != "leech" else 2064                     # Leech: 86 blocks, no tail
    pks, ws64 = [], []
    for i in range(4):
        if fmt == "bpdq":
            d = synth.bpdq(C, C, 9500 + i)
            pks.append(q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=ntok))
            ws64.append(obpdq.decode_f64(d["plane0"], d["plane1"], d["coef"]))
        elif fmt == "trellis":
            d = synth.trellis(C, C, 9510 + i)
            pks.append(q2.Packed(q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), ntok_max=ntok))
            ws64.append(otrellis.decode_f64(d["stream"], d["table"], d["scale"]))
        elif fmt == "leech":
            d = synth.leech(C, C, 9520 + i)
            pks.append(q2.Packed(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C), ntok_max=ntok))
            ws64.append(oleech.decode_f64(d["v"], d["scale"], d["tail"]))
        else:
            d = synth.fp16_dense(C, C, 9530 + i)
            pks.append(q2.Packed(q2.q2_pack_fp16(d["w"]), ntok_max=ntok))
            ws64.append(ofp16.decode_f64(d["w"]))
    x0 = synth.activations(ntok, C, 9540)
    bufs = [torch.from_numpy(x0).cuda()] + [torch.empty((ntok, C), dtype=torch.float16, device="cuda") for _ in pks]
    chain = q2.Chain([(p, bufs[i], bufs[i + 1]) for i, p in enumerate(pks)], ntok, 0)
    chain.run()
    torch.cuda.synchronize()
    x = x0
    for i, w in enumerate(ws64):
        y = bufs[i + 1].cpu().numpy()
        assert np.isfinite(y.astype(np.float32)).all(), f"GEMV {i}: non-finite outputs"
        ok = matvec.passes(y, matvec.gemv(w, x), matvec.abs_bound(w, x), 2e-3)
        assert ok.all(), f"GEMV {i}: {(~ok).sum()} outputs outside the tolerance"
        x = y
    assert q2.device_errors() == 0
