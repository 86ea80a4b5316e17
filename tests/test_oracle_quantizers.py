"""Invariant and brute-force pins of the quantizers (coverage bounds, code ranges, optimality)."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import quant
from oracle.nf4 import nf4_codebook
from synth import normal_weights


def _weights(seed, n, k, sigma=0.02):
    return normal_weights(seed, n, k, sigma, outlier_p=0.002, outlier_mult=20.0)


@pytest.mark.parametrize("fmt,g", [("INT4_SYM", 32), ("INT8_SYM", 128), ("INT4_SYM", 128)])
def test_symmetric_coverage_and_range(fmt, g):
    w = _weights(11, 24, 512)
    qz = quant.quantize(w, fmt, g)
    spec = quant.FORMATS[fmt]
    assert qz.codes.min() >= spec["qmin"] and qz.codes.max() <= spec["qmax"]
    s = np.repeat(qz.scale.astype(np.float64), g, axis=1)
    err = np.abs(w.astype(np.float64) - quant.dequant(qz).astype(np.float64))
    assert np.all(err <= s / 2)
    # the scale is the fp16 nearest to absmax / qmax
    absmax = np.abs(w.reshape(24, -1, g)).max(axis=2).astype(np.float64)
    assert np.all(np.abs(qz.scale.astype(np.float64) - absmax / spec["qmax"])
                  <= np.abs(np.nextafter(qz.scale, np.float16(np.inf)).astype(np.float64)
                            - qz.scale.astype(np.float64)) / 2 + 1e-30)


@pytest.mark.parametrize("fmt,g", [("INT4_ASYM", 128), ("INT4_ASYM", 32), ("INT2_ASYM", 64)])
def test_asymmetric_coverage_range_and_scale(fmt, g):
    w = _weights(12, 24, 512)
    qz = quant.quantize(w, fmt, g)
    levels = quant.FORMATS[fmt]["qmax"]
    assert qz.codes.min() >= 0 and qz.codes.max() <= levels
    z = qz.zero.astype(np.float64)
    assert np.all((z >= 0) & (z <= levels) & (z == np.rint(z)))
    wg = w.reshape(24, -1, g).astype(np.float64)
    span = np.maximum(wg.max(2), 0) - np.minimum(wg.min(2), 0)
    s = qz.scale.astype(np.float64)
    assert np.all(s * levels >= span)                                  # the grid covers the range
    prev = np.nextafter(qz.scale, np.float16(0)).astype(np.float64)
    assert np.all(prev * levels < span)                                # ... with the smallest such fp16
    err = np.abs(w.astype(np.float64) - quant.dequant(qz).astype(np.float64))
    assert np.all(err <= np.repeat(s, g, axis=1) / 2)


@pytest.mark.parametrize("fmt", ["INT4_SYM", "INT8_SYM", "INT4_ASYM", "INT2_ASYM"])
def test_integer_codes_are_nearest_brute_force(fmt):
    """For fixed metadata, no other code reconstructs any weight strictly closer (checked exactly)."""
    w = _weights(13, 3, 64)
    g = 32
    qz = quant.quantize(w, fmt, g)
    spec = quant.FORMATS[fmt]
    lo, hi = spec["qmin"], spec["qmax"]
    for r in range(3):
        for j in range(64):
            s = Fraction(float(qz.scale[r, j // g]))
            z = Fraction(float(qz.zero[r, j // g])) if qz.zero is not None else Fraction(0)
            wv = Fraction(float(w[r, j]))
            best = abs(wv - s * (int(qz.codes[r, j]) - z))
            for c in range(lo, hi + 1):
                assert abs(wv - s * (c - z)) >= best


def test_nf4_codes_are_nearest_with_lowest_index_ties():
    cb = nf4_codebook()
    w = _weights(14, 4, 128)
    qz = quant.quantize(w, "NF4", 64, codebook=cb)
    for r in range(4):
        for j in range(128):
            a = float(qz.scale[r, j // 64])
            ratio = float(w[r, j]) / a
            dist = [abs(ratio - float(c)) for c in cb]
            assert int(qz.codes[r, j]) == dist.index(min(dist))
    a = qz.scale.astype(np.float64)
    absmax = np.abs(w.reshape(4, -1, 64)).max(2)
    assert np.all(a == absmax.astype(np.float16).astype(np.float64))
    # reconstruction error bounded by half the widest codebook gap times a (plus the fp16 rounding of a)
    gap = np.max(np.diff(cb.astype(np.float64)))
    err = np.abs(w.astype(np.float64) - quant.dequant(qz).astype(np.float64))
    assert np.all(err <= np.repeat(a, 64, axis=1) * (gap / 2 + 2.0 ** -10))


def test_k4_ceilings_and_coverage():
    w = normal_weights(15, 16, 1024, 0.015)
    qz = quant.quantize(w, "K4", 256)
    assert qz.codes.min() >= 0 and qz.codes.max() <= 15
    assert qz.sc.max() <= 63 and qz.m.max() <= 63
    wb = w.reshape(16, 4, 8, 32).astype(np.float64)
    lo = np.minimum(wb.min(3), 0)
    hi = np.maximum(wb.max(3), 0)
    d = qz.d.astype(np.float64)[..., None]
    dmin = qz.dmin.astype(np.float64)[..., None]
    sc = qz.sc.astype(np.float64)
    m = qz.m.astype(np.float64)
    assert np.all(dmin * m >= -lo)                 # the min offset covers the most negative weight
    assert np.all(dmin * (m - 1) < -lo + (m == 0))  # ... and m is the smallest such code
    r = hi + dmin * m
    assert np.all(15 * d * sc >= r)
    assert np.all(15 * d * (sc - 1) < r + (sc == 0))
    exact = d[..., None] * sc[..., None] * qz.codes.reshape(16, 4, 8, 32) - (dmin * m)[..., None]
    assert np.all(np.abs(wb - exact) <= (d * sc)[..., None] / 2)


def test_zero_groups():
    w = np.zeros((2, 256), dtype=np.float32)
    for fmt, g in [("INT4_SYM", 32), ("INT8_SYM", 128), ("INT4_ASYM", 128), ("INT2_ASYM", 64)]:
        qz = quant.quantize(w, fmt, g)
        assert np.all(qz.scale == 0) and np.all(qz.codes == 0)
        assert np.all(quant.dequant(qz) == 0)
    cb = nf4_codebook()
    qz = quant.quantize(w, "NF4", 64, codebook=cb)
    assert np.all(cb[qz.codes] == 0) and np.all(quant.dequant(qz) == 0)
    qz = quant.quantize(w, "K4", 256)
    assert np.all(qz.d == 0) and np.all(qz.dmin == 0) and np.all(quant.dequant(qz) == 0)


def test_zero_nibble_layout():
    z = np.array([[1, 2, 3], [15, 0, 7]], dtype=np.uint8)
    p = quant.pack_zero_nibbles(z)
    assert p.tolist() == [[0x21, 0x03], [0x0F, 0x07]]
    assert np.array_equal(quant.unpack_zero_nibbles(p, 3), z)
    z2 = np.random.default_rng(0).integers(0, 16, (5, 32)).astype(np.uint8)
    assert np.array_equal(quant.unpack_zero_nibbles(quant.pack_zero_nibbles(z2), 32), z2)
