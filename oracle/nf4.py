"""The NF4 codebook: 16 standard-normal quantiles normalised to [-1, 1].

Source: "Ultra LLM Engine", section "Quantization" (row ``nf4``: NormalFloat4
with a QLoRA-style codebook); the workload definition says each 4-bit code
indexes a 16-entry fp32 codebook of standard-normal quantiles normalised to
[-1, 1], passed to the kernels as an input.

Construction (this library's own reading of "normal quantiles, asymmetric, with
an exact zero"): 8 positive values Phi^-1(1/2 + (i/8)(delta - 1/2)) for
i = 1..8, 7 negative values -Phi^-1(1/2 + (i/7)(delta - 1/2)) for i = 1..7, and
0; each side divided by its largest magnitude so the ends are exactly -1 and 1;
delta = 1 - 1/32.  Phi^-1 is Python's ``statistics.NormalDist().inv_cdf``.
Values are rounded to float32.  Both the oracle and the GPU path receive the
same 16 values, so parity does not depend on the table's provenance.
"""
from __future__ import annotations

from statistics import NormalDist

import numpy as np

DELTA = 1.0 - 1.0 / 32.0


def nf4_codebook(delta: float = DELTA) -> np.ndarray:
    """float32[16], ascending: 7 negative quantiles, 0, 8 positive quantiles; c[0] = -1, c[7] = 0, c[15] = 1."""
    inv = NormalDist().inv_cdf
    pos = [inv(0.5 + (i / 8.0) * (delta - 0.5)) for i in range(1, 9)]
    neg = [inv(0.5 + (i / 7.0) * (delta - 0.5)) for i in range(1, 8)]
    pos = [p / pos[-1] for p in pos]
    neg = [-v / neg[-1] for v in neg]
    vals = sorted(neg) + [0.0] + pos
    return np.asarray(vals, dtype=np.float64).astype(np.float32)
