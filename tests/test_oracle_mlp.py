"""Pins of the oracle's gated-MLP projection (oracle/mlp.py) against what mathematics fixes.

* silu against an independent high-precision evaluation (sympy, 40 digits) and the identity
  sigma(t) = (1 + tanh(t / 2)) / 2 computed through numpy's tanh;
* the odd-part identity silu(t) - silu(-t) = t, the closed form silu(ln 3) = (3/4) ln 3, the
  limits silu(0) = 0, silu(t) -> t (t -> +inf) and -> -0 (t -> -inf);
* the derivative bound |silu'| <= 1.1 the pass rule rests on;
* a hand-worked 1 x 32 case whose gate and up outputs are small integers (g = 1, u = 2), so
  h = 2 silu(1); swapping gate and up (h' = silu(2)) or dropping the gate (h'' = g * u) fails it;
* zero gate weights or zero up weights give h = 0 exactly.
"""
import math

import numpy as np
import pytest

from oracle import mlp, quant

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _sympy_silu(t):
    sympy = pytest.importorskip("sympy")
    v = sympy.Float(repr(float(t)), 40)
    return float(v / (1 + sympy.exp(-v)))


@pytest.mark.parametrize("t", [-30.0, -5.0, -1.0, -0.5, -1e-3, 0.0, 1e-3, 0.5, 1.0, 2.0, math.log(3.0), 5.0, 30.0])
def test_silu_against_high_precision(t):
    want = _sympy_silu(t)
    got = float(mlp.silu(np.array([t]))[0])
    assert got == pytest.approx(want, rel=2e-15, abs=1e-300)


def test_silu_against_the_tanh_form():
    t = np.random.default_rng(5).normal(0.0, 4.0, 10000)
    alt = t * 0.5 * (1.0 + np.tanh(0.5 * t))
    # 1 + tanh(t / 2) cancels for t << 0, so the alternative form carries an absolute error ~1e-16
    np.testing.assert_allclose(mlp.silu(t), alt, rtol=1e-14, atol=1e-15)


def test_silu_identities_and_limits():
    t = np.random.default_rng(6).normal(0.0, 3.0, 10000)
    np.testing.assert_allclose(mlp.silu(t) - mlp.silu(-t), t, rtol=1e-14, atol=1e-14)
    assert float(mlp.silu(np.array([math.log(3.0)]))[0]) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    assert float(mlp.silu(np.array([0.0]))[0]) == 0.0
    assert float(mlp.silu(np.array([50.0]))[0]) == pytest.approx(50.0, rel=1e-20)
    neg = float(mlp.silu(np.array([-1000.0]))[0])
    assert neg == 0.0 and math.copysign(1.0, neg) == -1.0


def test_silu_slope_bound():
    t = np.linspace(-20.0, 20.0, 400001)
    s = 1.0 / (1.0 + np.exp(-t))
    slope = s * (1.0 + t * (1.0 - s))                       # d/dt (t * sigma(t))
    assert np.abs(slope).max() <= mlp.SILU_SLOPE_MAX
    assert np.abs(slope).max() > 1.09                       # the bound is tight, not loose


def _int4_sym_row(codes):
    """One INT4_SYM row of 32 weights with scale 1 (fp16), so W_hat = codes exactly."""
    c = np.asarray(codes, dtype=np.int8).reshape(1, 32)
    return quant.Quantized("INT4_SYM", 32, c, scale=np.ones((1, 1), dtype=np.float16))


def test_hand_worked_gate_and_up():
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0], x[0, 5] = 1.0, -1.0
    gate = np.zeros(32, dtype=np.int8)
    gate[0], gate[5] = 3, 2                                  # g = 3 - 2 = 1
    up = np.zeros(32, dtype=np.int8)
    up[0], up[5] = 1, -1                                     # u = 1 + 1 = 2
    h, B = mlp.gated_quantized(x, _int4_sym_row(gate), _int4_sym_row(up))
    sigma1 = math.e / (1.0 + math.e)
    want = 2.0 * sigma1                                      # 2 silu(1) = 1.46211715726001
    assert h[0, 0] == pytest.approx(want, rel=1e-15)
    assert B[0, 0] >= abs(h[0, 0])
    ok = mlp.gated_error_ratio(np.array([[want]]), h, B)
    assert ok.max() <= 1e-12
    # planted mistakes: gate and up swapped (silu(2) * 1), the gate dropped (g * u)
    swapped, _ = mlp.gated_quantized(x, _int4_sym_row(up), _int4_sym_row(gate))
    assert mlp.gated_error_ratio(swapped, h, B).max() > 1.0
    assert mlp.gated_error_ratio(np.array([[1.0 * 2.0]]), h, B).max() > 1.0


def test_zero_gate_or_up_gives_zero():
    rng = np.random.default_rng(7)
    x = rng.normal(size=(3, 32)).astype(np.float32)
    w = _int4_sym_row(rng.integers(-8, 8, 32))
    zero = _int4_sym_row(np.zeros(32))
    h1, _ = mlp.gated_quantized(x, zero, w)
    h2, _ = mlp.gated_quantized(x, w, zero)
    assert np.all(h1 == 0.0) and np.all(h2 == 0.0)
