"""Dense fp16 control ("Unfolding the Leech Lattice", section 7: the byte
bound of the roofline is the fp16 control's measured bandwidth).  The weights
are the fp16 values themselves.

Test infrastructure only (see ``oracle/__init__.py``).
"""
from __future__ import annotations

import numpy as np


def decode_f64(w: np.ndarray) -> np.ndarray:
    return w.astype(np.float64)
