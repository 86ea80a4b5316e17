"""Plant plausible mistakes in the oracle (on the CPU) and check that its pins catch each one."""
import numpy as np
import pytest

from oracle import gemm, quant
from tests import test_oracle_gemm as tg
from tests import test_oracle_quantizers as tq
from tests import test_oracle_worked as tw


def _expect_failure(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_wrong_zero_point_sign_is_caught(monkeypatch):
    orig = quant.dequant

    def bad(qz):
        if qz.fmt in ("INT4_ASYM", "INT2_ASYM"):
            qz = quant.Quantized(qz.fmt, qz.group, qz.codes, scale=qz.scale,
                                 zero=(-qz.zero.astype(np.float64)).astype(np.float16))
        return orig(qz)
    monkeypatch.setattr(quant, "dequant", bad)
    _expect_failure(tw.test_worked_example, "INT4_ASYM")


def test_dropped_min_term_is_caught(monkeypatch):
    orig = quant.dequant

    def bad(qz):
        if qz.fmt == "K4":
            qz = quant.Quantized("K4", 256, qz.codes, d=qz.d, dmin=np.zeros_like(qz.dmin), sc=qz.sc, m=qz.m)
        return orig(qz)
    monkeypatch.setattr(quant, "dequant", bad)
    _expect_failure(tw.test_worked_example, "K4")


def test_round_half_away_from_zero_is_caught(monkeypatch):
    real_rint = np.rint
    monkeypatch.setattr(quant.np, "rint", lambda a: np.trunc(a + np.copysign(0.5, a)))
    try:
        _expect_failure(tw.test_worked_example, "INT4_SYM")
    finally:
        monkeypatch.setattr(quant.np, "rint", real_rint)


def test_transposed_operand_is_caught(monkeypatch):
    def bad(x, w_hat, rows=None):
        xd = np.asarray(x, dtype=np.float64)
        wd = np.asarray(w_hat, dtype=np.float64)
        y = (wd @ xd.T).T if xd.shape[1] == wd.shape[1] else None
        # a plausible slip: contract over the wrong axis of W when it is square-ish
        return (xd @ wd[:, : xd.shape[1]].T)[:, ::-1], np.abs(xd) @ np.abs(wd).T
    monkeypatch.setattr(gemm, "reference", bad)
    _expect_failure(tg.test_unit_scales_reduce_to_integer_matmul)


def test_scale_rounded_to_nearest_instead_of_up_is_caught(monkeypatch):
    monkeypatch.setattr(quant, "f16_up", lambda v: np.asarray(v, dtype=np.float64).astype(np.float16))
    monkeypatch.setattr(quant, "f16_next_up", lambda h: h)
    _expect_failure(tq.test_asymmetric_coverage_range_and_scale, "INT4_ASYM", 128)


def test_nf4_highest_index_tie_break_is_caught(monkeypatch):
    real_argmin = np.argmin

    def last_argmin(a, axis=None):
        a = np.asarray(a)
        if axis is None:
            return a.size - 1 - real_argmin(a.ravel()[::-1])
        return a.shape[axis] - 1 - real_argmin(np.flip(a, axis=axis), axis=axis)
    monkeypatch.setattr(quant.np, "argmin", last_argmin)
    try:
        _expect_failure(tw.test_worked_example, "NF4")
    finally:
        monkeypatch.setattr(quant.np, "argmin", real_argmin)
