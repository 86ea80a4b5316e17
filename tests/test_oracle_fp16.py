"""Pins for oracle.fp16 against an exhaustive table of fp16 values decoded from their bit fields."""
import numpy as np
import pytest

from oracle.fp16 import f16_rne, f16_up
from tests.exact import half_value

_POS = sorted({float(half_value(b)) for b in range(0x7C00)})     # every finite non-negative fp16
_POS_ARR = np.array(_POS)


def _nearest_even_ref(v: float) -> float:
    i = int(np.searchsorted(_POS_ARR, v))
    if i < len(_POS) and _POS[i] == v:
        return v
    lo, hi = _POS[i - 1], _POS[i]
    if v - lo < hi - v:
        return lo
    if hi - v < v - lo:
        return hi
    # tie: the one with an even significand (even bit pattern)
    lo_bits = int(np.float16(lo).view(np.uint16))
    return lo if lo_bits % 2 == 0 else hi


def test_f16_up_is_smallest_half_at_or_above():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.random(4000) * 2.0 ** rng.integers(-26, 15, 4000),
                        _POS_ARR[1:2000:7], np.array([0.0, 2.0 ** -24, 2.0 ** -14, 65504.0])])
    h = f16_up(v).astype(np.float64)
    for vi, hi in zip(v, h):
        i = int(np.searchsorted(_POS_ARR, vi))
        assert hi == _POS[i], (vi, hi, _POS[i])


def test_f16_rne_matches_table_including_ties_and_subnormals():
    rng = np.random.default_rng(8)
    v = rng.random(3000) * 2.0 ** rng.integers(-26, 15, 3000)
    mids = [(a + b) / 2 for a, b in zip(_POS[1:3000:13], _POS[2:3001:13])]      # exact ties
    v = np.concatenate([v, np.array(mids)])
    h = f16_rne(v).astype(np.float64)
    for vi, hi in zip(v, h):
        assert hi == _nearest_even_ref(float(vi)), vi


def test_f16_overflow_is_refused():
    with pytest.raises(AssertionError):
        f16_up(np.array([70000.0]))
