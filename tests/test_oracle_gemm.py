"""Pins of the oracle's dequantize-then-matmul, its bound and its pass rule."""
from fractions import Fraction

import numpy as np

from oracle import gemm, quant
from synth import activations, normal_weights


def test_reference_equals_exact_rational_sums():
    x = activations(21, 3, 96)
    w = normal_weights(21, 5, 96, 0.02)
    qz = quant.quantize(w, "INT4_ASYM", 32)
    w_hat = quant.dequant(qz)
    y, b = gemm.reference(x, w_hat)
    for m in range(3):
        for n in range(5):
            ex = sum(Fraction(float(x[m, k])) * Fraction(float(w_hat[n, k])) for k in range(96))
            eb = sum(abs(Fraction(float(x[m, k])) * Fraction(float(w_hat[n, k]))) for k in range(96))
            assert abs(Fraction(y[m, n]) - ex) <= eb * Fraction(96, 2 ** 52)
            assert abs(Fraction(b[m, n]) - eb) <= eb * Fraction(96, 2 ** 52)


def test_unit_scales_reduce_to_integer_matmul():
    """All s = 1, z = 0: y is the textbook integer GEMV of the codes (non-square, so a transpose fails)."""
    rng = np.random.default_rng(5)
    M, N, K = 3, 7, 64
    codes = rng.integers(-8, 8, (N, K)).astype(np.int8)
    xi = rng.integers(-20, 21, (M, K))
    qz = quant.Quantized("INT4_SYM", 32, codes, scale=np.ones((N, 2), dtype=np.float16))
    y, b = gemm.reference(xi.astype(np.float32), quant.dequant(qz))
    assert np.array_equal(y, (xi @ codes.astype(np.int64).T).astype(np.float64))
    assert np.array_equal(b, (np.abs(xi) @ np.abs(codes.astype(np.int64)).T).astype(np.float64))
    qz = quant.Quantized("INT4_ASYM", 32, (codes + 8).astype(np.int8), scale=np.ones((N, 2), dtype=np.float16),
                         zero=np.full((N, 2), 8, dtype=np.uint8))
    y2, _ = gemm.reference(xi.astype(np.float32), quant.dequant(qz))
    assert np.array_equal(y2, y)


def test_batched_rows_equal_single_row_calls():
    x = activations(22, 4, 256)
    w = normal_weights(22, 9, 256, 0.02)
    w_hat = quant.dequant(quant.quantize(w, "INT8_SYM", 128))
    y, b = gemm.reference(x, w_hat)
    for m in range(4):
        y1, b1 = gemm.reference(x[m:m + 1], w_hat)
        assert np.array_equal(y1[0], y[m]) and np.array_equal(b1[0], b[m])


def test_selected_rows_match_full():
    x = activations(23, 2, 128)
    w_hat = quant.dequant(quant.quantize(normal_weights(23, 40, 128, 0.02), "INT4_SYM", 32))
    y, b = gemm.reference(x, w_hat)
    rows = np.array([39, 0, 17])
    ys, bs = gemm.reference(x, w_hat, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(bs, b[:, rows])


def test_pass_rule():
    y_ref = np.array([[1.0, -2.0, 0.0]])
    b = np.array([[10.0, 4.0, 0.0]])
    at_limit = y_ref + np.array([[1e-2 + 1e-6, -(4e-3 + 1e-6), 1e-6]])
    r = gemm.error_ratio(at_limit, y_ref, b)
    assert np.allclose(r, 1.0)
    over = y_ref + np.array([[1.1e-2, 0.0, 0.0]])
    assert gemm.error_ratio(over, y_ref, b).max() > 1.0
