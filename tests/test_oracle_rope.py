"""Pins of the RMSNorm + RoPE oracle (oracle/rope.py) against closed forms and invariants.

* RMSNorm: a constant row gives gamma * c / sqrt(c^2 + eps); with eps = 0 the result does not depend
  on the row's scale; a sum in place of the mean fails the closed form;
* RoPE: position 0 is the identity; every rotated pair keeps its length; rotating by p1 then p2 equals
  rotating by p1 + p2; <rope(q, p1), rope(k, p2)> depends only on p1 - p2;
* a hand-worked head of 4 values at position 1 (angles 1 and 10000^-1/2): n = e_0 goes to
  (cos 1, 0, sin 1, 0); the interleaved pairing or a flipped sine sign gives something else.
"""
import math

import numpy as np
import pytest

from oracle import rope


def test_rmsnorm_closed_form_and_scale_invariance():
    c, eps = 0.75, 1e-5
    gamma = np.linspace(0.5, 2.0, 8)
    n = rope.rms_norm(np.full((1, 8), c), gamma, eps)
    np.testing.assert_allclose(n[0], gamma * c / math.sqrt(c * c + eps), rtol=1e-15)
    x = np.random.default_rng(1).normal(size=(3, 64))
    g = np.random.default_rng(2).normal(size=64)
    np.testing.assert_allclose(rope.rms_norm(7.5 * x, g, 0.0), rope.rms_norm(x, g, 0.0), rtol=1e-13)
    # planted: the sum of squares in place of the mean
    wrong = x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) * g
    assert not np.allclose(wrong, rope.rms_norm(x, g, 0.0))


def test_rope_identity_norm_and_composition():
    rng = np.random.default_rng(3)
    n = rng.normal(size=(5, 256))
    hd, base = 64, 10000.0
    np.testing.assert_allclose(rope.rotate(n, np.zeros(5), hd, base), n, rtol=0, atol=0)
    p = np.array([1, 7, 100, 4095, 65536])
    y = rope.rotate(n, p, hd, base)
    yh, nh = y.reshape(5, 4, hd), n.reshape(5, 4, hd)
    half = hd // 2
    np.testing.assert_allclose(yh[..., :half] ** 2 + yh[..., half:] ** 2, nh[..., :half] ** 2 + nh[..., half:] ** 2,
                               rtol=1e-12)
    p1, p2 = np.array([3, 11, 200, 7, 1]), np.array([5, 2, 1000, 9, 3])
    np.testing.assert_allclose(rope.rotate(rope.rotate(n, p1, hd, base), p2, hd, base),
                               rope.rotate(n, p1 + p2, hd, base), rtol=1e-9, atol=1e-12)


def test_rope_relative_position():
    rng = np.random.default_rng(4)
    q, k = rng.normal(size=(1, 128)), rng.normal(size=(1, 128))
    hd, base = 128, 500000.0
    dots = [float(np.sum(rope.rotate(q, np.array([p1]), hd, base) * rope.rotate(k, np.array([p1 - 17]), hd, base)))
            for p1 in (17, 40, 1000, 30000)]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


def test_hand_worked_head():
    n = np.array([[1.0, 0.0, 0.0, 0.0]])
    y = rope.rotate(n, np.array([1]), 4, 10000.0)
    want = np.array([[math.cos(1.0), 0.0, math.sin(1.0), 0.0]])
    np.testing.assert_allclose(y, want, rtol=1e-15, atol=1e-300)
    n2 = np.array([[0.0, 1.0, 0.0, 0.0]])              # the second pair: angle 10000^-1/2 = 0.01
    np.testing.assert_allclose(rope.rotate(n2, np.array([1]), 4, 10000.0), [[0.0, math.cos(0.01), 0.0, math.sin(0.01)]],
                               rtol=1e-15, atol=1e-300)
    ratio = rope.error_ratio(want, y, n, 4)
    assert ratio.max() < 1e-9
    # planted: interleaved pairs (0, 1) and a flipped sine both fail the pass rule
    inter = np.array([[math.cos(1.0), math.sin(1.0), 0.0, 0.0]])
    flipped = np.array([[math.cos(1.0), 0.0, -math.sin(1.0), 0.0]])
    assert rope.error_ratio(inter, y, n, 4).max() > 1.0
    assert rope.error_ratio(flipped, y, n, 4).max() > 1.0


def test_fused_is_norm_then_rotation():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(4, 256)).astype(np.float32)
    g = rng.normal(size=256)
    pos = np.array([0, 1, 31, 8191])
    y, n = rope.rmsnorm_rope(x, g, pos, 128, 1e-6, 10000.0)
    np.testing.assert_allclose(n, rope.rms_norm(x, g, 1e-6), rtol=0)
    np.testing.assert_allclose(y[0], n[0], rtol=0)        # position 0: the norm alone
    assert rope.error_ratio(y, y, n, 128).max() == 0.0


@pytest.mark.parametrize("hd", [2, 64, 128])
def test_partner_is_the_rotation_partner(hd):
    n = np.arange(2 * hd, dtype=np.float64).reshape(1, 2 * hd) + 1.0
    p = rope.partner(n, hd).reshape(2, hd)
    half = hd // 2
    assert np.array_equal(p[0, :half], n[0, half:hd]) and np.array_equal(p[1, half:], n[0, hd:hd + half])
