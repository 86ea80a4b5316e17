"""Brute-force pins of every decode: each code value x several fp16 scales, against exact rationals."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import quant
from oracle.nf4 import nf4_codebook
from tests.exact import half_value, round_to_f32

# fp16 bit patterns: 0, smallest subnormal, a mid subnormal, smallest normal, 0.125, 1, 0.02-ish, max
HALF_BITS = [0x0000, 0x0001, 0x0155, 0x0400, 0x3000, 0x3C00, 0x251F, 0x7BFF]


def _half(bits):
    return np.array([bits], dtype=np.uint16).view(np.float16)[0]


@pytest.mark.parametrize("fmt,lo,hi", [("INT4_SYM", -8, 7), ("INT8_SYM", -128, 127)])
def test_symmetric_decode_all_codes(fmt, lo, hi):
    codes = np.arange(lo, hi + 1, dtype=np.int64)
    g = 32
    reps = -(-len(codes) // g) * g
    q = np.resize(codes, reps).astype(np.int8).reshape(1, -1)
    for hb in HALF_BITS:
        G = q.shape[1] // g
        qz = quant.Quantized(fmt, g, q, scale=np.full((1, G), _half(hb), dtype=np.float16))
        w = quant.dequant(qz)[0]
        s = half_value(hb)
        for qi, wi in zip(q[0], w):
            assert float(wi) == round_to_f32(s * int(qi))


@pytest.mark.parametrize("fmt,levels", [("INT4_ASYM", 15), ("INT2_ASYM", 3)])
def test_asymmetric_decode_all_codes_and_zeros(fmt, levels):
    g = 32
    codes = np.resize(np.arange(levels + 1), g).astype(np.int8)
    for hb in HALF_BITS:
        for z in range(levels + 1):
            zero = np.array([[z]], dtype=np.uint8 if fmt == "INT4_ASYM" else np.float16)
            qz = quant.Quantized(fmt, g, codes[None, :].copy(),
                                 scale=np.array([[_half(hb)]], dtype=np.float16), zero=zero)
            w = quant.dequant(qz)[0]
            s = half_value(hb)
            for qi, wi in zip(codes, w):
                assert float(wi) == round_to_f32(s * (int(qi) - z))


def test_nf4_decode_all_codes():
    cb = nf4_codebook()
    codes = np.resize(np.arange(16), 64).astype(np.int8)
    for hb in HALF_BITS:
        qz = quant.Quantized("NF4", 64, codes[None, :].copy(),
                             scale=np.array([[_half(hb)]], dtype=np.float16), codebook=cb)
        w = quant.dequant(qz)[0]
        a = half_value(hb)
        for qi, wi in zip(codes, w):
            assert float(wi) == round_to_f32(a * Fraction(float(cb[qi])))


def test_k4_decode_all_scale_and_min_codes():
    """Every (sc, m) pair of 6-bit codes and every q, for (d, dmin) pairs including fp16 subnormals."""
    pairs = [(0x0155, 0x0001), (0x0400, 0x03FF), (0x1A3D, 0x2C00), (0x3C00, 0x0155)]
    n_sub = 64 * 64                                   # sub-block t carries sc = t // 64, m = t % 64
    n_sb = n_sub // 8
    t = np.arange(n_sub)
    sc = (t // 64).astype(np.uint8).reshape(1, n_sb, 8)
    m = (t % 64).astype(np.uint8).reshape(1, n_sb, 8)
    codes = (np.arange(n_sb * 256) % 16).astype(np.int8).reshape(1, -1)
    codes[0, ::32] = (t * 7) % 16                     # first weight of each sub-block cycles through q
    for db, mb in pairs:
        d, dmin = half_value(db), half_value(mb)
        qz = quant.Quantized("K4", 256, codes,
                             d=np.full((1, n_sb), _half(db), dtype=np.float16),
                             dmin=np.full((1, n_sb), _half(mb), dtype=np.float16),
                             sc=sc, m=m)
        w = quant.dequant(qz)[0]
        for ti in range(n_sub):
            j = ti * 32 + (ti % 32)
            exact = d * int(sc[0, ti // 8, ti % 8]) * int(codes[0, j]) - dmin * int(m[0, ti // 8, ti % 8])
            assert float(w[j]) == round_to_f32(exact), (ti, db, mb)
