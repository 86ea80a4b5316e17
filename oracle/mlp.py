"""The gated MLP's fused gate/up projection in float64: h = silu(x . W_gate^T) * (x . W_up^T).

Source: "Ultra LLM Engine", section "How the Engine Works": every decoder layer ends in a gated
MLP whose projections are quantized linear layers (the "quantized MLP projections" of the layer
diagram), and the checkpoint loader maps HF/Llama-style tensor names onto the model.  The page
does not spell the gate out; the plainest reading for a Llama-style decoder is the SiLU gate,
h = silu(g) * u with g = x . W_gate^T, u = x . W_up^T and silu(t) = t / (1 + e^-t), the input
of the down projection.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The device computes g and u in fp32 (the quantized linear layers' fp32 accumulation), evaluates
silu and the product in fp32 and rounds h to bf16 once.  Its error has three parts:
  * the errors of g and u, each within the linear layers' pass rule 1e-3 * b (b = sum |x * w_hat|),
    carried through h = silu(g) * u with |silu'(t)| <= 1.1 for every t:
        <= 1e-3 * (1.1 * b_g * |u| + |silu(g)| * b_u)   (to first order);
  * fp32 rounding of silu and of the product: a few units in 2^-24 relative to |h|;
  * the bf16 rounding of h: at most 2^-8 * |h| (half a unit in the last place of an 8-bit significand).
The pass rule therefore is |h - h_ref| <= 1e-3 * B + 2^-8 * |h_ref| + 1e-6 with
B = 1.1 * b_g * |u_ref| + |silu(g_ref)| * b_u: the second term is the output rounding, and the first
covers the fp32 errors (orders of magnitude below 1e-3 * B) together with the rounding's own slack.
"""
from __future__ import annotations

import numpy as np

from . import gemm, quant

REL_TOL = 1e-3
OUT_TOL = 2.0 ** -8
ABS_TOL = 1e-6
SILU_SLOPE_MAX = 1.1      # sup over t of |d/dt (t / (1 + e^-t))| = 1.0998...


def silu(t: np.ndarray) -> np.ndarray:
    """t / (1 + e^-t) in float64 (e^-t overflows to +inf for t < -709, giving -0: the limit)."""
    t = np.asarray(t, dtype=np.float64)
    with np.errstate(over="ignore"):
        return t / (1.0 + np.exp(-t))


def gated_reference(x: np.ndarray, w_gate_hat: np.ndarray, w_up_hat: np.ndarray):
    """(h_ref, B): float64 [m][n] gated output and the error scale B of the pass rule."""
    g, b_g = gemm.reference(x, w_gate_hat)
    u, b_u = gemm.reference(x, w_up_hat)
    sg = silu(g)
    h = sg * u
    B = SILU_SLOPE_MAX * b_g * np.abs(u) + np.abs(sg) * b_u
    return h, B


def gated_quantized(x: np.ndarray, qz_gate: "quant.Quantized", qz_up: "quant.Quantized"):
    """h_ref, B for x against the dequantized gate and up weights -- the whole oracle path."""
    return gated_reference(x, quant.dequant(qz_gate), quant.dequant(qz_up))


def gated_error_ratio(h_dev: np.ndarray, h_ref: np.ndarray, B: np.ndarray) -> np.ndarray:
    """|h_dev - h_ref| / (1e-3 * B + 2^-8 * |h_ref| + 1e-6); the pass rule is max <= 1."""
    hd = np.asarray(h_dev, dtype=np.float64)
    return np.abs(hd - h_ref) / (REL_TOL * B + OUT_TOL * np.abs(h_ref) + ABS_TOL)
