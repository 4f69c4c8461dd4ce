"""The allocation-free BPDQ entry point, q2_gemv_bpdq_noalloc.

It exists for callers that cannot allocate device memory when they run the
GEMV (code under CUDA stream capture, plugins whose host framework owns the
device memory, real-time loops that must not call the allocator): the split-K
accumulator words live in a scratch array owned by the library instead of a
caller-bound workspace.  This test calls it through the C ABI twice in a row,
on different activations, and checks each result against q2_gemv (the entry
point with a workspace) within the tolerance the parity tests use,
|y - y_ref| <= 2e-3 * sum_c |w x|.  It also checks that a problem larger than
the scratch is refused.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import synth
from oracle import bpdq as obpdq, matvec

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


def _noalloc(q2, pk, x, y):
    L = q2.load()
    st = L.q2_gemv_bpdq_noalloc(pk.h, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


@pytest.mark.parametrize("R,C,seed", [(4096, 4096, 7100), (70, 768, 7101)])
def test_noalloc_matches_workspace_entry_point(q2, R, C, seed):
    d = synth.bpdq(R, C, seed)
    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=1)
    w64 = obpdq.decode_f64(d["plane0"], d["plane1"], d["coef"])
    for call in range(2):                         # two calls in a row, different x
        x_np = synth.activations(1, C, seed + 10 * call + 1)
        x = torch.from_numpy(x_np).cuda()
        y_ref = pk.gemv(x)                        # q2_gemv with the caller's workspace
        y = torch.full((1, R), float("nan"), dtype=torch.float16, device="cuda")
        assert _noalloc(q2, pk, x, y) == 0
        torch.cuda.synchronize()
        bound = matvec.abs_bound(w64, x_np)
        diff = np.abs(y.cpu().numpy().astype(np.float64) - y_ref.cpu().numpy().astype(np.float64))
        assert np.all(diff <= TOL * bound), f"call {call}: max excess {(diff - TOL * bound).max():.3e}"
        # and against the oracle, with the same tolerance
        ok = matvec.passes(y.cpu().numpy(), matvec.gemv(w64, x_np), bound, TOL)
        assert ok.all()


def test_noalloc_refuses_problems_larger_than_the_scratch(q2):
    # 131104 rows x 8 bytes = 1,048,832 bytes > Q2_NOALLOC_SCRATCH_BYTES (1 MiB)
    R, C = 131104, 256
    d = synth.bpdq(R, C, 7200)
    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=1)
    x = torch.zeros((1, C), dtype=torch.float16, device="cuda")
    y = torch.zeros((1, R), dtype=torch.float16, device="cuda")
    assert _noalloc(q2, pk, x, y) == -11
    assert q2.q2_strerror(-11).startswith("problem larger than the built-in scratch")
