"""Pins of the W4A8 oracle (oracle/w4a8.py).

* activation quantization: codes in [-127, 127], the absmax element at +-127, |x - s_x q| <= s_x / 2
  (up to the fp32 quotient's rounding, checked against exact rationals), zero rows give zeros, each row
  its own scale (a per-tensor scale fails on rows of different magnitude);
* when every x is an exact multiple of a power-of-two scale (so quantization is lossless), the integer
  group sums reproduce the plain dequantize-then-matmul reference exactly, for all three formats;
* a hand-worked 1 x 8 case with a zero point.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import gemm, quant, w4a8


def test_activation_codes_range_and_error():
    rng = np.random.default_rng(21)
    x = rng.normal(size=(6, 512)).astype(np.float32)
    x[2] *= 1e-3
    x[4] = 0.0
    q, s = w4a8.quantize_activations(x)
    assert q.dtype == np.int8 and q.min() >= -127 and q.max() <= 127
    assert np.all(q[4] == 0) and s[4] == 0
    for m in (0, 1, 2, 3, 5):
        assert np.abs(q[m]).max() == 127
        sm = Fraction(float(s[m]))
        for k in range(0, 512, 7):
            exact = Fraction(float(x[m, k])) / sm
            # the fp32 quotient may round a value within 2^-23 of a half-integer to either side
            assert abs(exact - int(q[m, k])) <= Fraction(1, 2) + abs(exact) * Fraction(1, 2 ** 23)


def test_per_row_scales():
    x = np.array([[1.0, -0.5, 0.25, 0.0], [100.0, -50.0, 25.0, 0.0]], dtype=np.float32)
    q, s = w4a8.quantize_activations(x)
    assert q[0].tolist() == q[1].tolist() == [127, -64, 32, 0]      # 63.5 -> 64 and 31.75 -> 32 (nearest)
    assert s[1] == np.float32(100.0) / np.float32(127.0)
    # planted: one scale for the tensor would crush the first row's codes
    s_all = np.float32(100.0) / np.float32(127.0)
    assert np.rint(x[0] / s_all).tolist() != q[0].tolist()


@pytest.mark.parametrize("fmt,group", [("INT4_SYM", 32), ("INT4_ASYM", 128), ("INT8_SYM", 64)])
def test_lossless_activations_match_the_plain_reference(fmt, group):
    rng = np.random.default_rng(22)
    m, n, k = 3, 40, 512
    xq = rng.integers(-127, 128, (m, k))
    xq[:, 0] = 127                                                   # absmax 127 * 2^-7 in every row
    x = (xq * 2.0 ** -7).astype(np.float32)                          # s_x = 2^-7 exactly, x / s_x = xq exactly
    w = rng.normal(0, 0.02, (n, k)).astype(np.float32)
    qz = quant.quantize(w, fmt, group)
    y, b = w4a8.w4a8_reference(x, qz)
    y_plain, b_plain = gemm.reference(x, quant.dequant(qz))
    np.testing.assert_allclose(y, y_plain, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(b, b_plain, rtol=1e-12, atol=1e-15)


def test_hand_worked_with_zero_point():
    # x = [1, -1, 0.5, 0, 0, 0, 0, 0]: absmax 1, s_x = RN32(1/127), codes [127, -127, 64, 0, ...]
    x = np.zeros((1, 8), dtype=np.float32)
    x[0, :3] = [1.0, -1.0, 0.5]
    codes = np.array([[3, 10, 15, 0, 0, 0, 0, 0]], dtype=np.int8)
    qz = quant.Quantized("INT4_ASYM", 8, codes, scale=np.array([[0.25]], dtype=np.float16),
                         zero=np.array([[5]], dtype=np.uint8))
    y, _ = w4a8.w4a8_reference(x, qz)
    sx = float(np.float32(1.0) / np.float32(127.0))
    # I = 127 (3 - 5) - 127 (10 - 5) + 64 (15 - 5) + 5 * (0 - 5) * 0 = -254 - 635 + 640 = -249
    assert y[0, 0] == pytest.approx(sx * 0.25 * -249, rel=1e-15)
