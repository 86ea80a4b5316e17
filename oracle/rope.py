"""RMSNorm followed by rotary position embedding (RoPE), in float64.

Source: "Ultra LLM Engine", section "Fused Kernels" (a fused "RMSNorm followed by RoPE" operation) and
section "How the Engine Works" (each layer applies RMSNorm and rotary position embeddings before the
quantized attention projections).  The page gives no formulas; the plainest reading, the one of the
Llama-style models its loader targets:

  RMSNorm   n[m][j] = x[m][j] / sqrt(mean_j(x[m][j]^2) + eps) * gamma[j]   over the row's D values;
  RoPE      each consecutive block of head_dim values of a row is one head; within it, value i and value
            i + head_dim/2 (i < head_dim/2) are rotated by the angle pos[m] * base^(-2 i / head_dim):
              y_i          = n_i cos(a) - n_{i+h/2} sin(a)
              y_{i + h/2}  = n_{i+h/2} cos(a) + n_i sin(a)
            (the "rotate half" pairing; pos[m] is the row's position).

A row can be a token's whole hidden vector (D = hidden size) or one head's vector (D = head_dim, the
per-head query/key norm of some Llama-style families): the same definition covers both.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The device computes in fp32 from bf16 x and gamma with cos/sin from a table rounded to fp32, and rounds
y to bf16 once.  Its error: fp32 reduction and normalisation (relative well below 1e-5 of |n|), the
table's rounding (2^-24) and the bf16 rounding of y (at most 2^-8 |y|).  Pass rule:
    |y - y_ref| <= 2^-8 * |y_ref| + 1e-4 * (|n_i| + |n_partner|) + 1e-6.
"""
from __future__ import annotations

import numpy as np

OUT_TOL = 2.0 ** -8
REL_TOL = 1e-4
ABS_TOL = 1e-6


def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """n = x / sqrt(mean(x^2) + eps) * gamma over each row, float64."""
    xd = np.asarray(x, dtype=np.float64)
    ms = np.mean(xd * xd, axis=-1, keepdims=True)
    return xd / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)


def rope_angles(pos: np.ndarray, head_dim: int, base: float) -> np.ndarray:
    """a[m][i] = pos[m] * base^(-2 i / head_dim), i < head_dim / 2, float64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv = base ** (-2.0 * i / head_dim)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]


def rotate(n: np.ndarray, pos: np.ndarray, head_dim: int, base: float) -> np.ndarray:
    """Rotate-half RoPE of every head_dim block of each row of n by the row's position."""
    m, d = n.shape
    assert head_dim % 2 == 0 and d % head_dim == 0
    a = rope_angles(pos, head_dim, base)                    # [m][h/2]
    c, s = np.cos(a)[:, None, :], np.sin(a)[:, None, :]
    nh = n.reshape(m, d // head_dim, head_dim)
    lo, hi = nh[..., : head_dim // 2], nh[..., head_dim // 2:]
    y = np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)
    return y.reshape(m, d)


def partner(n: np.ndarray, head_dim: int) -> np.ndarray:
    """|n| of each value's rotation partner (i <-> i + head_dim/2 within its head)."""
    m, d = n.shape
    nh = np.abs(n).reshape(m, d // head_dim, head_dim)
    half = head_dim // 2
    return np.concatenate([nh[..., half:], nh[..., :half]], axis=-1).reshape(m, d)


def rmsnorm_rope(x, gamma, pos, head_dim: int, eps: float, base: float):
    """(y_ref, n): the fused output and the normalised input it rotates, both float64 [m][d]."""
    n = rms_norm(x, gamma, eps)
    return rotate(n, pos, head_dim, base), n


def error_ratio(y_dev, y_ref, n, head_dim: int) -> np.ndarray:
    """|y_dev - y_ref| / (2^-8 |y_ref| + 1e-4 (|n_i| + |n_partner|) + 1e-6); the pass rule is max <= 1."""
    yd = np.asarray(y_dev, dtype=np.float64)
    scale = np.abs(n) + partner(n, head_dim)
    return np.abs(yd - y_ref) / (OUT_TOL * np.abs(y_ref) + REL_TOL * scale + ABS_TOL)
