"""Dequantize-then-matmul in float64, the per-element error bound, and the pass rule.

Source: "Ultra LLM Engine", section "Fused Kernels": a dequantized-weight GEMV
for single-token decode and a dequantized-weight GEMM for batched decode.  The
oracle computes the plain definition

    y_ref[m, n] = sum_k x[m, k] * W_hat[n, k]        (float64)
    b[m, n]     = sum_k |x[m, k] * W_hat[n, k]|      (float64)

x holds bf16 values and W_hat float32 values, so every product is exact in
float64 (8 + 24 significand bits) and the only error is float64 accumulation
(about k * 2^-53 relative to b).  A device result y (bf16, fp32 accumulation)
passes when |y - y_ref| <= 1e-3 * b + 1e-6 for every element.
"""
from __future__ import annotations

import numpy as np

from . import quant

REL_TOL = 1e-3
ABS_TOL = 1e-6


def reference(x: np.ndarray, w_hat: np.ndarray, rows: np.ndarray | None = None):
    """(y_ref, b), both float64 [m][n] (or [m][len(rows)] for the selected rows of W_hat)."""
    xd = np.asarray(x, dtype=np.float32).astype(np.float64)
    w = np.asarray(w_hat, dtype=np.float32)
    if rows is not None:
        w = w[np.asarray(rows)]
    n = w.shape[0]
    y = np.empty((xd.shape[0], n), dtype=np.float64)
    b = np.empty_like(y)
    ax = np.abs(xd)
    step = max(1, (1 << 24) // max(1, w.shape[1]))
    for r0 in range(0, n, step):
        wd = w[r0:r0 + step].astype(np.float64)
        y[:, r0:r0 + step] = xd @ wd.T
        b[:, r0:r0 + step] = ax @ np.abs(wd).T
    return y, b


def error_ratio(y_dev: np.ndarray, y_ref: np.ndarray, b: np.ndarray,
                rel: float = REL_TOL, abs_: float = ABS_TOL) -> np.ndarray:
    """|y_dev - y_ref| / (rel * b + abs) elementwise; the pass rule is max <= 1."""
    yd = np.asarray(y_dev, dtype=np.float64)
    return np.abs(yd - y_ref) / (rel * b + abs_)


def quantized_gemm(x: np.ndarray, qz: "quant.Quantized", rows=None):
    """y_ref, b for x against dequant(qz) -- the whole oracle path in one call."""
    return reference(x, quant.dequant(qz), rows=rows)
