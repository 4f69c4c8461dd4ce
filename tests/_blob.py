"""Host-side readers of q2 blobs for the layout tests (no GPU needed)."""
import numpy as np

HEADER = np.dtype([
    ("magic", "<u4"), ("version", "<u4"), ("fmt", "<i4"), ("R", "<i4"), ("C", "<i4"), ("Rpad", "<i4"),
    ("nslice", "<i4"), ("nblock", "<i4"), ("tail", "<i4"), ("tailpad", "<i4"), ("nexc", "<u4"),
    ("inv_sqrt8", "<f4"), ("total", "<u8"), ("off", "<u8", (8,)), ("len", "<u8", (8,)),
    ("layout", "<i4"), ("reserved", "<i4"),
])


def header(blob: np.ndarray):
    return np.frombuffer(blob[:HEADER.itemsize].tobytes(), dtype=HEADER)[0]


def section(blob: np.ndarray, i: int) -> np.ndarray:
    h = header(blob)
    return blob[int(h["off"][i]): int(h["off"][i]) + int(h["len"][i])]


def unrotate_planes(sec: np.ndarray, nplanes: int, R: int, S: int, Rpad: int) -> np.ndarray:
    """Item stream -> canonical plane bytes [nplanes][R][S*32]."""
    nrb = Rpad // 32
    items = sec.reshape(S, nrb, 2 * nplanes, 32, 16)         # slice, rb, chunk, lane, byte
    out = np.zeros((nplanes, Rpad, S * 32), dtype=np.uint8)
    lane = np.arange(32)
    for k in range(2 * nplanes):
        for q in range(16):
            P = (k & 1) * 16 + q
            beta = (P + lane) & 31                            # [32]
            for s in range(S):
                vals = items[s, :, k, :, q]                   # [nrb][32]
                rows = (np.arange(nrb)[:, None] * 32 + lane[None, :])
                out[k >> 1, rows, s * 32 + beta[None, :]] = vals
    return out[:, :R]
