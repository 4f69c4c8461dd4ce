"""Host-side tests of the C ABI (no GPU): the library loads, exports what
include/q2.h declares, the packers lay out the canonical content as the
device kernels expect it, and bad arguments return the documented status."""
import ctypes
import os
import re
import shutil

import numpy as np
import pytest

import synth
from oracle import bpdq as obpdq
from tests import _blob

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q2():
    import dequant_gemv_q2_gb300 as m
    if not os.path.exists(m.lib_path()):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("libq2.so not built and nvcc not available")
        m._build.build()
    m.load()
    return m


def test_exports_every_declared_symbol(q2):
    hdr = open(os.path.join(ROOT, "include", "q2.h")).read()
    names = set(re.findall(r"\b(q2_[a-z0-9_]+)\s*\(", hdr))
    assert {"q2_gemv", "q2_bind", "q2_pack_bpdq", "q2_pack_trellis", "q2_pack_leech"} <= names
    L = ctypes.CDLL(q2.lib_path())
    for n in sorted(names):
        assert hasattr(L, n), n
    assert set(q2.EXPORTS) == names


def test_bpdq_layout_and_value_table(q2):
    R, C = 70, 768                       # ragged rows, three groups
    d = synth.bpdq(R, C, seed=21)
    blob = q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"])
    h = _blob.header(blob)
    assert (h["fmt"], h["R"], h["C"], h["Rpad"], h["nslice"]) == (1, R, C, 96, 3)
    planes = _blob.unrotate_planes(_blob.section(blob, 0), 2, R, 3, 96)
    assert np.array_equal(planes[0], d["plane0"]) and np.array_equal(planes[1], d["plane1"])
    vt = _blob.section(blob, 3).view(np.uint16).reshape(3, 96, 4)[:, :R]
    # the table entry for code k equals the oracle's canonical fp16 weight
    for k in range(4):
        p0 = np.full_like(d["plane0"], 0xFF if k & 1 else 0)
        p1 = np.full_like(d["plane1"], 0xFF if k & 2 else 0)
        w = obpdq.decode_fp16(p0, p1, d["coef"])               # [R][C]
        assert np.array_equal(vt[:, :, k].T.view(np.float16), w[:, ::256])
    c01 = _blob.section(blob, 1).view(np.uint16).reshape(3, 96, 2)[:, :R]
    off = _blob.section(blob, 2).view(np.uint16).reshape(3, 96)[:, :R]
    assert np.array_equal(c01, d["coef"][:, :, :2].view(np.uint16))
    assert np.array_equal(off, d["coef"][:, :, 2].view(np.uint16))


def test_trellis_layout(q2):
    R, C = 33, 512
    d = synth.trellis(R, C, seed=5)
    blob = q2.q2_pack_trellis(d["stream"], d["table"], d["scale"])
    h = _blob.header(blob)
    sec = _blob.section(blob, 0).reshape(2, 2, 4, 32, 16)       # seg, rb, chunk, lane, bytes
    for r in (0, 1, 31, 32):
        rb, l = divmod(r, 32)
        for s in range(2):
            lane_bytes = np.concatenate([sec[s, rb, k, l] for k in range(4)])
            nib = np.empty(128, dtype=np.uint8)
            nib[0::2] = lane_bytes & 15
            nib[1::2] = lane_bytes >> 4
            seg = d["stream"][r, s]
            sym = np.empty(128, dtype=np.uint8)
            sym[0::2] = seg & 15
            sym[1::2] = seg >> 4
            assert np.array_equal(nib, sym[::-1])      # nibble n = symbol 127 - n
    assert np.array_equal(_blob.section(blob, 1).view(np.float16).reshape(4096, 2), d["table"])
    assert h["nslice"] == 2


def test_leech_layout_roundtrip(q2):
    R, C = 40, 24 * 30 + 8
    d = synth.leech(R, C, seed=77)
    v = d["v"].copy()
    v[3, 5] = 0
    v[3, 5, 7] = 8                       # +8 goes to the exception channel
    v[10, 29] = 0
    v[10, 29, [0, 1]] = [-8, 0]
    blob = q2.q2_pack_leech(v, d["tail"], d["scale"], C)
    h = _blob.header(blob)
    S = h["nslice"]
    planes = _blob.unrotate_planes(_blob.section(blob, 0), 3, R, S, int(h["Rpad"]))
    bits = [np.unpackbits(planes[q], axis=1, bitorder="little") for q in range(3)]
    par = _blob.section(blob, 1).view(np.uint16).reshape(S, -1)
    nb = C // 24
    u = bits[0] + 2 * bits[1].astype(np.int64) - 4 * bits[2].astype(np.int64)
    rec = np.zeros((R, nb, 24), dtype=np.int64)
    for b in range(nb):
        sb = 24 * b // 256
        first = (256 * sb + 23) // 24
        p = (par[sb, :R] >> (b - first)) & 1
        rec[:, b] = p[:, None] + 2 * u[:, 24 * b: 24 * b + 24]
    ptr = _blob.section(blob, 4).view(np.uint32)
    col = _blob.section(blob, 5).view(np.uint32)
    assert h["nexc"] == 1 and ptr[3] == 0 and ptr[4] == 1 and col[0] == 5 * 24 + 7
    rec.reshape(R, -1)[3, col[0]] = 8
    assert np.array_equal(rec, v.astype(np.int64))
    tail = _blob.section(blob, 3).view(np.float16).reshape(-1, int(h["tailpad"]))[:R, :8]
    assert np.array_equal(tail, d["tail"])


def test_leech_offset_binary_layout_roundtrip(q2):
    """The second Leech layout: four planes of c = (v - p)/2 + 4, no exceptions."""
    R, C = 40, 24 * 30 + 8
    d = synth.leech(R, C, seed=78)
    v = d["v"].copy()
    v[3, 5] = 0
    v[3, 5, 7] = 8                       # +8 is code 8 (plane 3), not an exception
    v[10, 29] = 0
    v[10, 29, [0, 1]] = [-8, 0]          # -8 is code 0
    blob = q2.q2_pack_leech(v, d["tail"], d["scale"], C, q2.LEECH_OFFSET4)
    h = _blob.header(blob)
    assert h["layout"] == 1 and h["nexc"] == 0 and h["version"] == 2
    S = h["nslice"]
    planes = _blob.unrotate_planes(_blob.section(blob, 0), 4, R, S, int(h["Rpad"]))
    bits = [np.unpackbits(planes[q], axis=1, bitorder="little").astype(np.int64) for q in range(4)]
    code = bits[0] + 2 * bits[1] + 4 * bits[2] + 8 * bits[3]
    par = _blob.section(blob, 1).view(np.uint16).reshape(S, -1)
    nb = C // 24
    rec = np.zeros((R, nb, 24), dtype=np.int64)
    for b in range(nb):
        sb = 24 * b // 256
        first = (256 * sb + 23) // 24
        p = (par[sb, :R] >> (b - first)) & 1
        rec[:, b] = p[:, None] + 2 * (code[:, 24 * b: 24 * b + 24] - 4)
    assert np.array_equal(rec, v.astype(np.int64))
    assert (code[:, nb * 24:] == 4).all()                        # outside the blocks: code 4, the code of 0
    # 4 planes + parity + scale + tail: one bit per weight more than the three-plane layout
    b3 = q2.q2_pack_leech(v, d["tail"], d["scale"], C)
    assert _blob.header(b3)["len"][0] * 4 == h["len"][0] * 3
    L = q2.load()
    n = ctypes.c_size_t(0)
    assert L.q2_pack_leech(None, None, None, R, C, ctypes.c_float(0.35), 2, None, ctypes.byref(n)) == -1


def test_status_codes(q2):
    L = q2.load()
    n = ctypes.c_size_t(0)
    assert L.q2_pack_bpdq(None, None, None, 4, 300, None, ctypes.byref(n)) == -2      # C % 256
    assert L.q2_pack_trellis(None, None, None, 0, 256, None, ctypes.byref(n)) == -2
    assert L.q2_pack_fp16(None, 4, 12, None, ctypes.byref(n)) == -2
    assert L.q2_pack_noweights(64, 512, None, None) == -1
    d = synth.bpdq(32, 256, seed=1)
    blob = q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"])
    small = np.zeros(16, dtype=np.uint8)
    n = ctypes.c_size_t(16)
    p0 = np.ascontiguousarray(d["plane0"])
    st = L.q2_pack_bpdq(p0.ctypes.data, p0.ctypes.data, d["coef"].ctypes.data, 32, 256,
                        small.ctypes.data, ctypes.byref(n))
    assert st == -10 and n.value == blob.size
    bad = blob.copy()
    bad[0] ^= 1
    h = ctypes.c_void_p()
    fake_dev = ctypes.c_void_p(1 << 20)                    # never dereferenced by q2_bind
    assert L.q2_bind(bad.ctypes.data, fake_dev, ctypes.byref(h)) == -6
    assert L.q2_bind(blob.ctypes.data, ctypes.c_void_p((1 << 20) + 16), ctypes.byref(h)) == -3
    assert L.q2_bind(blob.ctypes.data, fake_dev, ctypes.byref(h)) == 0
    ws = ctypes.c_size_t(0)
    assert L.q2_workspace_bytes(h, 1, ctypes.byref(ws)) == 0
    assert ws.value == 1 * 32 * 8                             # one 64-bit accumulator word per (token, row)
    assert L.q2_workspace_bytes(h, 3, ctypes.byref(ws)) == 0 and ws.value == 3 * 32 * 8
    # tensor-core path, one slice: no K split, the launch writes y itself and needs no workspace
    assert L.q2_workspace_bytes(h, 7, ctypes.byref(ws)) == 0 and ws.value == 0

    assert L.q2_workspace_bytes(h, 65, ctypes.byref(ws)) == -5
    x = ctypes.c_void_p(1 << 21)
    assert L.q2_gemv(2, h, x, x, 1, None) == -4                              # fmt mismatch
    assert L.q2_gemv(1, h, x, x, 0, None) == -5                              # ntok
    assert L.q2_gemv(1, h, ctypes.c_void_p((1 << 21) + 2), x, 1, None) == -3  # alignment
    assert L.q2_gemv(1, h, x, x, 1, None) == -7                              # no workspace
    assert L.q2_strerror(-7) == b"workspace missing or too small"
    # the chain checks every link before it launches anything
    fmts = (ctypes.c_int * 2)(1, 1)
    hs = (ctypes.c_void_p * 2)(h.value, h.value)
    xs = (ctypes.c_void_p * 2)(1 << 21, 1 << 21)
    assert L.q2_gemv_chain(0, None, None, None, None, 1, 2, None) == 0                 # empty chain
    assert L.q2_gemv_chain(2, fmts, hs, xs, xs, 1, 5, None) == -1                      # lookahead > 4
    assert L.q2_gemv_chain(2, fmts, hs, xs, xs, 1, -1, None) == -1
    assert L.q2_gemv_chain(2, fmts, None, xs, xs, 1, 2, None) == -1
    fmts[1] = 2
    assert L.q2_gemv_chain(2, fmts, hs, xs, xs, 1, 2, None) == -4                      # fmt of link 1
    fmts[1] = 1
    assert L.q2_gemv_chain(2, fmts, hs, xs, xs, 1, 2, None) == -7                      # no workspace
    L.q2_unbind(h)


def test_rotation_split_and_argument_checks(q2):
    # q2_rotate_split follows the page's examples; q2_rotate validates every
    # argument before it touches the device (the pointers below are never read)
    assert q2.q2_rotate_split(5120) == (1024, 5)
    assert q2.q2_rotate_split(6144) == (2048, 3)
    assert q2.q2_rotate_split(17408) == (1024, 17)
    assert q2.q2_rotate_split(4096) == (2048, 2)
    L = q2.load()
    a, b = ctypes.c_int(), ctypes.c_int()
    assert L.q2_rotate_split(1000, ctypes.byref(a), ctypes.byref(b)) == -2          # not a multiple of 1024
    assert L.q2_rotate_split(4096, None, ctypes.byref(b)) == -1
    x, y, s, q = (ctypes.c_void_p(1 << k) for k in (21, 22, 23, 24))
    assert L.q2_rotate(None, y, 1, 4096, 2048, s, q, None) == -1                    # null x
    assert L.q2_rotate(x, y, 1, 4096, 2048, None, q, None) == -1                    # null signs
    assert L.q2_rotate(x, y, 0, 4096, 2048, s, q, None) == -5                       # ntok
    assert L.q2_rotate(x, y, 65, 4096, 2048, s, q, None) == -5
    assert L.q2_rotate(x, y, 1, 4096, 1000, s, q, None) == -2                       # nh not a power of two
    assert L.q2_rotate(x, y, 1, 4097, 1024, s, q, None) == -2                       # C % nh
    assert L.q2_rotate(x, y, 1, 64 * 33, 64, s, q, None) == -2                      # nq = 33 > 32
    assert L.q2_rotate(x, y, 1, 2048 * 32, 2048, s, q, None) == -2                  # C over the maximum
    assert L.q2_rotate(x, y, 1, 4096, 1024, s, None, None) == -1                    # nq = 4 needs Q
    assert L.q2_rotate(x, x, 1, 4096, 4096, s, None, None) == -1                    # in place


_PACK_SCRIPT = r"""
import hashlib, sys
sys.path.insert(0, {root!r})
import numpy as np
import dequant_gemv_q2_gb300 as q2
import synth
out = []
d = synth.bpdq(70, 768, 5)
out.append(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]))
d = synth.trellis(70, 512, 6)
out.append(q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]))
d = synth.leech(70, 1040, 7)
out.append(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], 1040))
out.append(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], 1040, layout=q2.LEECH_OFFSET4))
d = synth.fp16_dense(70, 1032, 8)
out.append(q2.q2_pack_fp16(d["w"]))
out.append(q2.q2_pack_noweights(70, 768))
print(" ".join(hashlib.sha256(np.ascontiguousarray(b).tobytes()).hexdigest() for b in out))
"""


def test_packed_blobs_are_identical_across_processes(q2):
    """A blob is a pure function of its canonical inputs: every byte,
    alignment padding included, is the same in two separate processes (so a
    blob written on one machine matches one packed on another)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = _PACK_SCRIPT.format(root=root)
    runs = [subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, cwd=root)
            for _ in range(2)]
    for r in runs:
        assert r.returncode == 0, r.stderr[-2000:]
    assert runs[0].stdout.split() == runs[1].stdout.split()
    assert len(runs[0].stdout.split()) == 6
