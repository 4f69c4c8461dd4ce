"""Fused dequantize-plus-matvec over packed ~2-bit weights on GB300.

Thin ctypes binding of ``libq2.so`` (``include/q2.h``): the functions below
carry the C names and only marshal arguments; every step of y = W x runs in
the library's CUDA kernels.  PyTorch is used for device memory and streams.
Importing works without a GPU; calling a compute entry point without the
built library raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

FP16, BPDQ, TRELLIS, LEECH, NOWEIGHTS = 0, 1, 2, 3, 4
FMT_NAMES = {FP16: "fp16", BPDQ: "bpdq", TRELLIS: "trellis", LEECH: "leech", NOWEIGHTS: "noweights"}
MAX_NTOK = 64
INV_SQRT8_F32 = float(np.float32(1.0 / np.sqrt(8.0)))

_lib = None


class Q2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {q2_strerror(status)} ({status})")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libq2.so (build it first if asked); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise RuntimeError(f"libq2.so not built ({_build.LIB}); run __graft_entry__.build()")
        _build.build()
    L = ctypes.CDLL(_build.LIB)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    psz = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "q2_pack_fp16": [vp, i32, i32, vp, psz],
        "q2_pack_bpdq": [vp, vp, vp, i32, i32, vp, psz],
        "q2_pack_trellis": [vp, vp, vp, i32, i32, vp, psz],
        "q2_pack_leech": [vp, vp, vp, i32, i32, ctypes.c_float, i32, vp, psz],
        "q2_pack_noweights": [i32, i32, vp, psz],
        "q2_bind": [vp, vp, ctypes.POINTER(vp)],
        "q2_workspace_bytes": [vp, i32, psz],
        "q2_set_workspace": [vp, vp, sz],
        "q2_info": [vp, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)],
        "q2_bytes": [vp, i32, psz],
        "q2_gemv": [i32, vp, vp, vp, i32, vp],
        "q2_decode_bytes": [vp, psz],
        "q2_decode": [vp, vp, vp],
        "q2_gemv_chain": [i32, vp, vp, vp, vp, i32, i32, vp],
        "q2_gemv_bpdq_noalloc": [vp, vp, vp, vp],
        "q2_device_errors": [ctypes.POINTER(ctypes.c_uint)],
        "q2_debug_wait_limit": [ctypes.c_longlong],
        "q2_rotate": [vp, vp, i32, i32, i32, vp, vp, vp],
        "q2_rotate_split": [i32, ctypes.POINTER(i32), ctypes.POINTER(i32)],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = i32
    L.q2_unbind.argtypes = [vp]
    L.q2_unbind.restype = None
    L.q2_strerror.argtypes = [i32]
    L.q2_strerror.restype = ctypes.c_char_p
    _lib = L
    return L


EXPORTS = ["q2_pack_fp16", "q2_pack_bpdq", "q2_pack_trellis", "q2_pack_leech", "q2_pack_noweights",
           "q2_bind", "q2_unbind", "q2_workspace_bytes", "q2_set_workspace", "q2_info", "q2_bytes",
           "q2_gemv", "q2_gemv_chain", "q2_decode_bytes", "q2_decode", "q2_strerror", "q2_gemv_bpdq_noalloc",
           "q2_device_errors", "q2_debug_wait_limit", "q2_rotate", "q2_rotate_split"]


def q2_strerror(status: int) -> str:
    try:
        return load().q2_strerror(int(status)).decode()
    except Exception:  # library missing: still give a message
        return f"status {status}"


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _check(st: int, where: str) -> None:
    if st != 0:
        raise Q2Error(st, where)


def _pack(fn, args, where: str) -> np.ndarray:
    L = load()
    n = ctypes.c_size_t(0)
    _check(getattr(L, fn)(*args, None, ctypes.byref(n)), where)
    out = np.zeros(n.value, dtype=np.uint8)
    _check(getattr(L, fn)(*args, _ptr(out), ctypes.byref(n)), where)
    return out


def q2_pack_fp16(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.float16)
    R, C = w.shape
    return _pack("q2_pack_fp16", [_ptr(w.view(np.uint16)), R, C], "q2_pack_fp16")


def q2_pack_bpdq(plane0: np.ndarray, plane1: np.ndarray, coef: np.ndarray) -> np.ndarray:
    p0 = np.ascontiguousarray(plane0, dtype=np.uint8)
    p1 = np.ascontiguousarray(plane1, dtype=np.uint8)
    cf = np.ascontiguousarray(coef, dtype=np.float16)
    R, C = p0.shape[0], p0.shape[1] * 8
    return _pack("q2_pack_bpdq", [_ptr(p0), _ptr(p1), _ptr(cf.view(np.uint16)), R, C], "q2_pack_bpdq")


def q2_pack_trellis(stream: np.ndarray, table: np.ndarray, scale: np.ndarray) -> np.ndarray:
    st = np.ascontiguousarray(stream, dtype=np.uint8)
    tb = np.ascontiguousarray(table, dtype=np.float16)
    sc = np.ascontiguousarray(scale, dtype=np.float16)
    R, C = st.shape[0], st.shape[1] * 256
    return _pack("q2_pack_trellis", [_ptr(st), _ptr(tb.view(np.uint16)), _ptr(sc.view(np.uint16)), R, C],
                 "q2_pack_trellis")


LEECH_PLANES3, LEECH_OFFSET4 = 0, 1


def q2_pack_leech(v: np.ndarray, tail: np.ndarray, scale: np.ndarray, C: int, layout: int = LEECH_PLANES3) -> np.ndarray:
    vv = np.ascontiguousarray(v, dtype=np.int8)
    tl = np.ascontiguousarray(tail, dtype=np.float16)
    sc = np.ascontiguousarray(scale, dtype=np.float16)
    R = vv.shape[0]
    tptr = _ptr(tl.view(np.uint16)) if tl.size else None
    return _pack("q2_pack_leech", [_ptr(vv), tptr, _ptr(sc.view(np.uint16)), R, C,
                                   ctypes.c_float(INV_SQRT8_F32), int(layout)], "q2_pack_leech")


def q2_pack_noweights(R: int, C: int) -> np.ndarray:
    return _pack("q2_pack_noweights", [R, C], "q2_pack_noweights")


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def device_errors() -> int:
    """The tensor-core kernels' device error word (then cleared); 0 is normal."""
    v = ctypes.c_uint(0)
    _check(load().q2_device_errors(ctypes.byref(v)), "q2_device_errors")
    return v.value


def debug_wait_limit(polls: int) -> None:
    """Test hook: limit the tensor-core kernel's stage waits to `polls` polls (0 = normal)."""
    _check(load().q2_debug_wait_limit(int(polls)), "q2_debug_wait_limit")


class Packed:
    """A packed matrix bound to its device copy (and a split-K workspace).

    ``blob`` is the host blob from a ``q2_pack_*`` call.  The device copy and
    the workspace are torch tensors owned by this object.
    """

    def __init__(self, blob: np.ndarray, device="cuda", ntok_max: int = MAX_NTOK, workspace=None):
        import torch
        L = load()
        self.blob = blob
        self.dev = torch.from_numpy(blob).to(device)
        assert self.dev.data_ptr() % 256 == 0
        h = ctypes.c_void_p()
        _check(L.q2_bind(_ptr(blob), ctypes.c_void_p(self.dev.data_ptr()), ctypes.byref(h)), "q2_bind")
        self.h = h
        f, R, C = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check(L.q2_info(h, ctypes.byref(f), ctypes.byref(R), ctypes.byref(C)), "q2_info")
        self.fmt, self.R, self.C = f.value, R.value, C.value
        self.ws = None
        # the workspace of every call up to ntok_max tokens (the paths differ by token count)
        need = max(self.workspace_bytes(t) for t in range(1, int(ntok_max) + 1))
        if workspace is not None:
            self.set_workspace(workspace)
        elif need:
            self.set_workspace(torch.zeros(need, dtype=torch.uint8, device=device))

    def workspace_bytes(self, ntok: int) -> int:
        n = ctypes.c_size_t(0)
        _check(load().q2_workspace_bytes(self.h, int(ntok), ctypes.byref(n)), "q2_workspace_bytes")
        return n.value

    def set_workspace(self, ws) -> None:
        self.ws = ws
        _check(load().q2_set_workspace(self.h, ctypes.c_void_p(ws.data_ptr()), ws.numel()), "q2_set_workspace")

    def bytes_read(self, ntok: int = 1) -> int:
        n = ctypes.c_size_t(0)
        _check(load().q2_bytes(self.h, int(ntok), ctypes.byref(n)), "q2_bytes")
        return n.value

    def gemv(self, x, y=None, stream=None, fmt=None):
        """y[ntok][R] = x[ntok][C] @ W^T through q2_gemv (asynchronous)."""
        import torch
        if x.dim() == 1:
            x = x.view(1, -1)
        ntok = x.shape[0]
        if y is None:
            y = torch.empty((ntok, self.R), dtype=torch.float16, device=x.device)
        st = load().q2_gemv(self.fmt if fmt is None else int(fmt), self.h, ctypes.c_void_p(x.data_ptr()),
                            ctypes.c_void_p(y.data_ptr()), ntok, _stream_ptr(stream))
        _check(st, "q2_gemv")
        return y

    def decode(self, stream=None):
        """Canonical decode on the device (a uint8 tensor of q2_decode_bytes)."""
        import torch
        n = ctypes.c_size_t(0)
        _check(load().q2_decode_bytes(self.h, ctypes.byref(n)), "q2_decode_bytes")
        out = torch.zeros(n.value, dtype=torch.uint8, device=self.dev.device)
        _check(load().q2_decode(self.h, ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream)), "q2_decode")
        return out

    def close(self) -> None:
        if getattr(self, "h", None):
            load().q2_unbind(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def q2_gemv(fmt: int, packed: Packed, x, y, ntok: int, stream=None) -> int:
    """The C entry point with its own argument order (status returned)."""
    return load().q2_gemv(int(fmt), packed.h, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                          int(ntok), _stream_ptr(stream))


class Chain:
    """A decode step's chain of GEMVs run through q2_gemv_chain.

    ``links`` is a list of (Packed, x, y) with device fp16 tensors x [ntok][C]
    and y [ntok][R]; the pointer arrays are built once, so ``run`` only makes
    the one C call (and may be captured in a CUDA graph).
    """

    def __init__(self, links, ntok: int, lookahead: int = 2):
        n = len(links)
        self.links = list(links)            # keeps the tensors alive
        self.ntok, self.lookahead = int(ntok), int(lookahead)
        self._fmt = (ctypes.c_int * n)(*[p.fmt for p, _, _ in links])
        self._h = (ctypes.c_void_p * n)(*[p.h.value for p, _, _ in links])
        self._x = (ctypes.c_void_p * n)(*[x.data_ptr() for _, x, _ in links])
        self._y = (ctypes.c_void_p * n)(*[y.data_ptr() for _, _, y in links])

    def run(self, stream=None) -> None:
        st = load().q2_gemv_chain(len(self.links), self._fmt, self._h, self._x, self._y, self.ntok, self.lookahead,
                                  _stream_ptr(stream))
        _check(st, "q2_gemv_chain")


def q2_rotate_split(C: int) -> tuple:
    """(nh, nq) of the page's examples: nh = 2048 if it divides C, else 1024."""
    nh, nq = ctypes.c_int(), ctypes.c_int()
    _check(load().q2_rotate_split(int(C), ctypes.byref(nh), ctypes.byref(nq)), "q2_rotate_split")
    return nh.value, nq.value


def q2_rotate(x, x_rot, ntok: int, C: int, nh: int, signs, q, stream=None) -> int:
    """The C entry point (status returned): x_rot = (H (x) Q)(S x) per token."""
    return load().q2_rotate(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(x_rot.data_ptr()), int(ntok), int(C),
                            int(nh), ctypes.c_void_p(signs.data_ptr()),
                            ctypes.c_void_p(q.data_ptr()) if q is not None else None, _stream_ptr(stream))


class Rotation:
    """The activation rotation of one input width, x_rot = (H (x) Q)(S x).

    ``signs``: uint8 [ceil(C/8)] column sign bits; ``q``: fp32 [nq][nq]
    (None when nq == 1).  Both are copied to the device once.
    """

    def __init__(self, signs: np.ndarray, q, nh: int, C: int, device="cuda"):
        import torch
        self.C, self.nh = int(C), int(nh)
        self.signs = torch.from_numpy(np.ascontiguousarray(signs, dtype=np.uint8)).to(device)
        self.q = None if q is None else torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).to(device)

    def apply(self, x, out=None, stream=None):
        """Rotate x [ntok][C] (fp16, device) into a new or given fp16 tensor (asynchronous)."""
        import torch
        if x.dim() == 1:
            x = x.view(1, -1)
        if out is None:
            out = torch.empty_like(x)
        _check(q2_rotate(x, out, x.shape[0], self.C, self.nh, self.signs, self.q, stream), "q2_rotate")
        return out
