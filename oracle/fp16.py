"""fp16 rounding helpers (float64 in, float16 out).

The workload definitions store scales as fp16.  Symmetric scales are rounded to
nearest-even; asymmetric and two-level scales are rounded toward +inf so that
the quantization grid always covers the group's range (the reading adopted for
"(max-min)/15": a scale rounded down could leave the extreme weight one code
outside the range).
"""
from __future__ import annotations

import numpy as np

F16_MAX = 65504.0


def f16_rne(v) -> np.ndarray:
    """Round float64 values to the nearest fp16, ties to even (NumPy converts float64 -> float16 directly)."""
    v = np.asarray(v, dtype=np.float64)
    h = v.astype(np.float16)
    assert np.all(np.isfinite(h)), "fp16 overflow"
    return h


def f16_up(v) -> np.ndarray:
    """Smallest fp16 value >= v, for finite non-negative float64 v."""
    v = np.asarray(v, dtype=np.float64)
    assert np.all(v >= 0.0)
    h = v.astype(np.float16)
    low = h.astype(np.float64) < v
    if np.any(low):
        h = np.where(low, np.nextafter(h, np.float16(np.inf)), h)
    assert np.all(np.isfinite(h)), "fp16 overflow"
    assert np.all(h.astype(np.float64) >= v)
    return h.astype(np.float16)


def f16_next_up(h) -> np.ndarray:
    """The next fp16 value above h."""
    h = np.asarray(h, dtype=np.float16)
    return np.nextafter(h, np.float16(np.inf)).astype(np.float16)
