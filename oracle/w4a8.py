"""W4A8: dynamic per-row int8 quantization of the activations and integer dot products, in float64.

Source: "Ultra LLM Engine", section "Quantized Model": linear layers are stored as quantized weights and
the activations are dynamically quantized for the GEMV/GEMM paths.  The page gives no formulas; the
plainest reading, symmetric per-row int8:

  s_x[m]    = absmax_k |x[m][k]| / 127, one fp32 division (a zero row has s_x = 0 and codes 0);
  xq[m][k]  = clamp(RNE(x[m][k] / s_x[m]), -127, 127), the quotient an fp32 division (the decision of
              an integer code is taken in the kernel's precision, so the two sides agree bit for bit);
  y[m][n]   = s_x[m] * sum_g s[n][g] * I[m][n][g],   I = sum_{k in g} xq[m][k] * (q[n][k] - z[n][g])

with the weight's own codes q, zero points z and fp16 scales s (INT4_SYM, INT4_ASYM, INT8_SYM: z = 0 for
the symmetric formats).  I is an exact integer; the device forms it with 4-way int8 dot products (dp4a).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The device's y differs from y_ref by fp32 rounding of the per-group products and their sum (a few
hundred units in 2^-24 of b' = s_x * sum_g |s_g| * sum_k |xq * (q - z)| at most) and the bf16 rounding
of y (2^-8 |y|).  Pass rule: |y - y_ref| <= 1e-4 * b' + 2^-8 * |y_ref| + 1e-6.
"""
from __future__ import annotations

import numpy as np

from . import quant

REL_TOL = 1e-4
OUT_TOL = 2.0 ** -8
ABS_TOL = 1e-6


def quantize_activations(x: np.ndarray):
    """(xq int8 [m][k], s_x float32 [m]) per the rule above."""
    xf = np.asarray(x, dtype=np.float32)
    absmax = np.max(np.abs(xf), axis=1)
    s = (absmax / np.float32(127.0)).astype(np.float32)             # fp32 division
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    quot = (xf / safe[:, None]).astype(np.float32)                  # fp32 division
    q = np.clip(np.rint(quot), -127, 127)
    q = np.where(s[:, None] > 0, q, 0.0)
    return q.astype(np.int8), s


def _codes_and_zeros(qz: "quant.Quantized"):
    q = qz.codes.astype(np.int64)
    n, k = q.shape
    G = k // qz.group
    if qz.fmt == "INT4_ASYM":
        z = qz.zero.astype(np.int64)
    elif qz.fmt in ("INT4_SYM", "INT8_SYM"):
        z = np.zeros((n, G), dtype=np.int64)
    else:
        raise ValueError(f"W4A8 takes INT4_SYM, INT4_ASYM or INT8_SYM weights, not {qz.fmt}")
    return q, z


def w4a8_reference(x: np.ndarray, qz: "quant.Quantized"):
    """(y_ref, b') float64 [m][n]: the integer-sum form of the quantized-activation product and its scale."""
    xq, sx = quantize_activations(x)
    q, z = _codes_and_zeros(qz)
    n, k = q.shape
    g = qz.group
    G = k // g
    s = qz.scale.astype(np.float64)                                  # [n][G]
    xg = xq.astype(np.int64).reshape(-1, G, g)                        # [m][G][g]
    y = np.zeros((xq.shape[0], n))
    b = np.zeros_like(y)
    step = max(1, (1 << 22) // max(1, k))
    for r0 in range(0, n, step):
        qg = q[r0:r0 + step].reshape(-1, G, g) - z[r0:r0 + step][:, :, None]   # [n'][G][g] integer (q - z)
        I = np.einsum("mgk,ngk->mng", xg, qg)                         # exact integer group sums
        A = np.einsum("mgk,ngk->mng", np.abs(xg), np.abs(qg))
        y[:, r0:r0 + step] = np.einsum("mng,ng->mn", I.astype(np.float64), s[r0:r0 + step])
        b[:, r0:r0 + step] = np.einsum("mng,ng->mn", A.astype(np.float64), np.abs(s[r0:r0 + step]))
    sxd = sx.astype(np.float64)[:, None]
    return y * sxd, b * sxd


def error_ratio(y_dev, y_ref, b) -> np.ndarray:
    """|y_dev - y_ref| / (1e-4 b' + 2^-8 |y_ref| + 1e-6); the pass rule is max <= 1."""
    yd = np.asarray(y_dev, dtype=np.float64)
    return np.abs(yd - y_ref) / (REL_TOL * b + OUT_TOL * np.abs(y_ref) + ABS_TOL)
