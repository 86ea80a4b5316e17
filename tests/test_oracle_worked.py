"""Pin the oracle's quantizers, dequantizers and product to hand-worked examples (tests/golden)."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import gemm, quant
from tests.golden_io import read_blocks

BLOCKS = read_blocks("worked_examples.txt")


def _f32(vals):
    return np.array([float(v) for v in vals], dtype=np.float32)


@pytest.mark.parametrize("fmt", ["INT4_SYM", "INT4_ASYM", "INT8_SYM", "INT2_ASYM", "NF4", "K4"])
def test_worked_example(fmt):
    b = BLOCKS[fmt]
    group = int(b["group"][0])
    w = _f32(b["w"])[None, :]
    x = _f32(b["x"])[None, :]
    cb = _f32(b["codebook"]) if "codebook" in b else None
    qz = quant.quantize(w, fmt, group, codebook=cb)
    assert qz.codes[0].tolist() == [int(v) for v in b["q"]]
    if fmt == "K4":
        assert Fraction(float(qz.d[0, 0])) == b["d"][0]
        assert Fraction(float(qz.dmin[0, 0])) == b["dmin"][0]
        assert qz.sc[0, 0].tolist() == [int(v) for v in b["sc"]]
        assert qz.m[0, 0].tolist() == [int(v) for v in b["m"]]
    else:
        assert Fraction(float(qz.scale[0, 0])) == b["scale"][0]
        if "zero" in b:
            assert float(qz.zero[0, 0]) == float(b["zero"][0])
    w_hat = quant.dequant(qz)
    assert [Fraction(float(v)) for v in w_hat[0]] == b["w_hat"]
    y, bound = gemm.reference(x, w_hat)
    assert Fraction(float(y[0, 0])) == b["y"][0]
    assert bound[0, 0] == pytest.approx(float(sum(abs(xi * wi) for xi, wi in zip(b["x"], b["w_hat"]))))
