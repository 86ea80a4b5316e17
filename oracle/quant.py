"""Quantizers and dequantizers of the six weight formats (CPU, float64 arithmetic).

Source: "Ultra LLM Engine", section "Quantization" -- the ``int`` scheme is
group-wise uniform INT-N for 2, 4 and 8 bits, the ``nf4`` scheme uses a
QLoRA-style NormalFloat4 codebook, and both expose dequantization helpers for
the fused kernels.  The concrete formulas follow the workload definitions the
library is measured on; each open point is resolved in the docstring that
makes it.

Weights W are n x k float32 (k contiguous, a linear layer's weight); groups run
along k.  Codes are returned as int8 n x k; metadata in natural row-major order
([n][k/group]).  Dequantized weights W_hat are float32 and are the correctly
rounded value of the exact real-valued formula (for the integer formats the
formula is exact in float32).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

from .fp16 import f16_rne, f16_up, f16_next_up

F64 = np.float64

# code ranges the quantizers emit; the decoders accept the full b-bit range
FORMATS = {
    "INT4_SYM": dict(bits=4, qmin=-8, qmax=7),
    "INT4_ASYM": dict(bits=4, qmin=0, qmax=15),
    "INT8_SYM": dict(bits=8, qmin=-127, qmax=127),
    "INT2_ASYM": dict(bits=2, qmin=0, qmax=3),
    "NF4": dict(bits=4, qmin=0, qmax=15),
    "K4": dict(bits=4, qmin=0, qmax=15),
}
K4_SUPER = 256   # weights per super-block
K4_SUB = 32      # weights per sub-block (8 per super-block)


@dataclass
class Quantized:
    fmt: str
    group: int
    codes: np.ndarray                      # int8 [n][k]
    scale: Optional[np.ndarray] = None     # fp16 [n][k/group]: s (INT*), absmax a (NF4)
    zero: Optional[np.ndarray] = None      # INT4_ASYM: uint8 [n][k/group] in 0..15; INT2_ASYM: fp16 [n][k/group]
    codebook: Optional[np.ndarray] = None  # NF4: float32[16]
    d: Optional[np.ndarray] = None         # K4: fp16 [n][k/256]
    dmin: Optional[np.ndarray] = None      # K4: fp16 [n][k/256]
    sc: Optional[np.ndarray] = None        # K4: uint8 [n][k/256][8] in 0..63
    m: Optional[np.ndarray] = None         # K4: uint8 [n][k/256][8] in 0..63


def _two_sum_exact(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """a + b in float64, asserting (Knuth's TwoSum error term is 0) that the sum was exact."""
    s = a + b
    bb = s - a
    err = (a - (s - bb)) + (b - bb)
    assert np.all(err == 0.0), "float64 sum not exact: exponent span too large for the oracle"
    return s


def _groups(w: np.ndarray, group: int) -> np.ndarray:
    n, k = w.shape
    assert k % group == 0, "k must be a multiple of the group size"
    return np.asarray(w, dtype=np.float32).reshape(n, k // group, group).astype(F64)


def quantize_sym(w: np.ndarray, group: int, fmt: str) -> Quantized:
    """Symmetric INT-N: s = fp16_RNE(absmax / qmax), q = clamp(RNE(w / s), qmin, qmax), W_hat = s * q.

    qmax = 7 (INT4_SYM, codes [-8, 7]) or 127 (INT8_SYM, codes [-127, 127]).
    Open points, plainest reading: w / s is rounded half-to-even (NumPy ``rint``,
    the rounding of the NumPy engine on the page); a group of zeros has s = 0
    and q = 0.  The quotient is formed in float64 from the fp16 scale.
    """
    spec = FORMATS[fmt]
    qmin, qmax = spec["qmin"], spec["qmax"]
    wg = _groups(w, group)
    absmax = np.max(np.abs(wg), axis=2)
    s = f16_rne(absmax / qmax)
    sf = s.astype(F64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(sf > 0.0, wg / np.where(sf > 0.0, sf, 1.0), 0.0)
    q = np.clip(np.rint(r), qmin, qmax)
    return Quantized(fmt, group, q.reshape(w.shape).astype(np.int8), scale=s)


def quantize_asym(w: np.ndarray, group: int, fmt: str) -> Quantized:
    """Asymmetric INT-N with integer zero point, L = 2^bits - 1 levels.

    mn = min(min(w_g), 0), mx = max(max(w_g), 0);  s = fp16 of (mx - mn) / L
    rounded toward +inf;  z = RNE(-mn / s);  q = clamp(RNE(w / s) + z, 0, L);
    W_hat = s * (q - z).

    Open points, plainest reading: the range includes 0 (so z is a code, and
    it equals the literal (max - min) / L whenever a group has both signs);
    the scale rounds up so every weight of the group is within s/2 of its
    reconstruction; an all-zero group has s = 0, z = 0, q = 0.  INT4_ASYM
    stores z as an unsigned 4-bit integer, INT2_ASYM stores z in fp16.
    """
    spec = FORMATS[fmt]
    levels = spec["qmax"]
    wg = _groups(w, group)
    mn = np.minimum(np.min(wg, axis=2), 0.0)
    mx = np.maximum(np.max(wg, axis=2), 0.0)
    span = _two_sum_exact(mx, -mn)
    s = f16_up(span / levels)
    short = s.astype(F64) * levels < span          # float64 quotient rounded below an fp16 value
    if np.any(short):
        s = np.where(short, f16_next_up(s), s).astype(np.float16)
    sf = s.astype(F64)
    pos = sf > 0.0
    safe = np.where(pos, sf, 1.0)
    z = np.where(pos, np.rint(-mn / safe), 0.0)
    assert np.all((z >= 0) & (z <= levels))
    r = np.where(pos[..., None], wg / safe[..., None], 0.0)
    q = np.clip(np.rint(r) + z[..., None], 0, levels)
    q = np.where(pos[..., None], q, 0.0)
    zero = z.astype(np.uint8) if fmt == "INT4_ASYM" else z.astype(np.float16)
    return Quantized(fmt, group, q.reshape(w.shape).astype(np.int8), scale=s, zero=zero)


def quantize_nf4(w: np.ndarray, group: int, codebook: np.ndarray) -> Quantized:
    """NF4: a = fp16_RNE(absmax_g);  q = first index minimising |w / a - c[i]| (float64);  W_hat = RN32(a * c[q]).

    The codebook c (16 float32 values, ascending) is an input.  Open points,
    plainest reading: ties go to the lower index; a group of zeros has a = 0
    and takes the index of the codebook's zero entry.
    """
    c = np.asarray(codebook, dtype=np.float32).astype(F64)
    assert c.shape == (16,)
    wg = _groups(w, group)
    a = f16_rne(np.max(np.abs(wg), axis=2))
    af = a.astype(F64)[..., None]
    zero_idx = int(np.argmin(np.abs(c)))
    n = wg.shape[0]
    q = np.empty(wg.shape, dtype=np.int8)
    step = max(1, (1 << 22) // max(1, wg.shape[1] * wg.shape[2]))
    for r0 in range(0, n, step):
        blk = wg[r0:r0 + step]
        ab = af[r0:r0 + step]
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = blk / np.where(ab > 0.0, ab, 1.0)
        dist = np.abs(ratio[..., None] - c)           # [rows][G][g][16]
        idx = np.argmin(dist, axis=-1)                # first minimum = lowest index on ties
        idx = np.where(ab > 0.0, idx, zero_idx)
        q[r0:r0 + step] = idx.astype(np.int8)
    return Quantized("NF4", group, q.reshape(w.shape), scale=a,
                     codebook=np.asarray(codebook, dtype=np.float32).copy())


def quantize_k4(w: np.ndarray) -> Quantized:
    """Two-level INT4: 256-weight super-blocks, 8 sub-blocks of 32, W_hat = d*sc_j*q - dmin*m_j.

    d and dmin are fp16 per super-block, sc_j and m_j are 6-bit codes per
    sub-block, q are 4-bit codes.  The workload defines only the
    reconstruction formula; this min/max quantizer with ceilings is the
    library's own, chosen so every weight is within d*sc_j/2 of its exact
    reconstruction:

      lo_j = min(min(w_j), 0), hi_j = max(max(w_j), 0)
      dmin = fp16 toward +inf of max_j(-lo_j) / 63,   m_j = ceil(-lo_j / dmin)
      r_j  = hi_j + dmin*m_j
      d    = fp16 toward +inf of max_j(r_j) / 945,    sc_j = ceil(r_j / (15 d))
      q    = clamp(RNE((w + dmin*m_j) / (d*sc_j)), 0, 15)  (q = 0 where d*sc_j = 0)

    Each ceiling is checked exactly (the products are exact in float64) and
    bumped by one where the float64 quotient rounded below the true value.
    """
    n, k = w.shape
    assert k % K4_SUPER == 0, "k must be a multiple of 256"
    S = k // K4_SUPER
    wb = np.asarray(w, dtype=np.float32).reshape(n, S, 8, K4_SUB).astype(F64)
    lo = np.minimum(np.min(wb, axis=3), 0.0)
    hi = np.maximum(np.max(wb, axis=3), 0.0)
    neg = -lo
    negmax = np.max(neg, axis=2)
    dmin = f16_up(negmax / 63.0)
    short = dmin.astype(F64) * 63.0 < negmax
    if np.any(short):
        dmin = np.where(short, f16_next_up(dmin), dmin).astype(np.float16)
    dminf = dmin.astype(F64)[..., None]
    safe = np.where(dminf > 0.0, dminf, 1.0)
    m = np.where(dminf > 0.0, np.ceil(neg / safe), 0.0)
    m = np.where(m * dminf < neg, m + 1.0, m)
    assert np.all((m >= 0) & (m <= 63))
    off = dminf * m                                   # exact: 11-bit x 6-bit
    r = _two_sum_exact(hi, off)
    R = np.max(r, axis=2)
    d = f16_up(R / 945.0)
    short = d.astype(F64) * 945.0 < R
    if np.any(short):
        d = np.where(short, f16_next_up(d), d).astype(np.float16)
    df = d.astype(F64)[..., None]
    unit = 15.0 * df
    safe = np.where(unit > 0.0, unit, 1.0)
    sc = np.where(unit > 0.0, np.ceil(r / safe), 0.0)
    sc = np.where(unit * sc < r, sc + 1.0, sc)
    assert np.all((sc >= 0) & (sc <= 63))
    ds = df * sc                                      # exact: 11-bit x 6-bit
    num = _two_sum_exact(wb, off[..., None])
    dss = np.where(ds > 0.0, ds, 1.0)[..., None]
    q = np.where(ds[..., None] > 0.0, np.clip(np.rint(num / dss), 0, 15), 0.0)
    return Quantized("K4", K4_SUPER, q.reshape(n, k).astype(np.int8),
                     d=d, dmin=dmin, sc=sc.astype(np.uint8), m=m.astype(np.uint8))


def quantize(w: np.ndarray, fmt: str, group: int, codebook: Optional[np.ndarray] = None) -> Quantized:
    """Quantize W (n x k float32) in ``fmt`` with groups of ``group`` along k."""
    if fmt in ("INT4_SYM", "INT8_SYM"):
        return quantize_sym(w, group, fmt)
    if fmt in ("INT4_ASYM", "INT2_ASYM"):
        return quantize_asym(w, group, fmt)
    if fmt == "NF4":
        return quantize_nf4(w, group, codebook)
    if fmt == "K4":
        assert group == K4_SUPER
        return quantize_k4(w)
    raise ValueError(fmt)


def dequant(qz: Quantized) -> np.ndarray:
    """W_hat (n x k float32): the correctly rounded value of the format's reconstruction formula.

    INT*_SYM: s*q; INT*_ASYM: s*(q - z); NF4: RN32(a * c[q]); K4: RN32(d*sc*q - dmin*m).
    The integer formats are exact in float32; NF4's product is exact in
    float64 (11 + 24 bits) and rounded once; K4's difference is exact in
    float64 (asserted) and rounded once.
    """
    n, k = qz.codes.shape
    q = qz.codes.astype(F64)
    if qz.fmt == "K4":
        S = k // K4_SUPER
        qb = q.reshape(n, S, 8, K4_SUB)
        df = qz.d.astype(F64)[..., None, None]
        dminf = qz.dmin.astype(F64)[..., None, None]
        a = df * qz.sc.astype(F64)[..., None] * qb          # exact: <= 21 bits
        b = dminf * qz.m.astype(F64)[..., None]             # exact: <= 17 bits
        wh = _two_sum_exact(a, -np.broadcast_to(b, a.shape))
        return wh.reshape(n, k).astype(np.float32)
    g = qz.group
    qg = q.reshape(n, k // g, g)
    s = qz.scale.astype(F64)[..., None]
    if qz.fmt in ("INT4_SYM", "INT8_SYM"):
        wh = s * qg
    elif qz.fmt in ("INT4_ASYM", "INT2_ASYM"):
        wh = s * (qg - qz.zero.astype(F64)[..., None])
    elif qz.fmt == "NF4":
        c = qz.codebook.astype(F64)
        wh = s * c[qz.codes.reshape(n, k // g, g).astype(np.int64)]
    else:
        raise ValueError(qz.fmt)
    return wh.reshape(n, k).astype(np.float32)


def pack_zero_nibbles(z: np.ndarray) -> np.ndarray:
    """INT4_ASYM zero points in the caller-facing layout: two per byte, [n][ceil(G/2)], low nibble = even group."""
    z = np.asarray(z, dtype=np.uint8)
    n, G = z.shape
    out = np.zeros((n, (G + 1) // 2), dtype=np.uint8)
    out[:, :] = z[:, 0::2] & 0xF
    out[:, : G // 2] |= (z[:, 1::2] & 0xF) << 4
    return out


def unpack_zero_nibbles(zp: np.ndarray, G: int) -> np.ndarray:
    """Inverse of :func:`pack_zero_nibbles`."""
    zp = np.asarray(zp, dtype=np.uint8)
    z = np.empty((zp.shape[0], G), dtype=np.uint8)
    z[:, 0::2] = zp[:, : (G + 1) // 2] & 0xF
    z[:, 1::2] = zp[:, : G // 2] >> 4
    return z
