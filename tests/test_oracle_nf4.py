"""Pin the NF4 codebook construction to scipy's normal quantile function (an independent library routine)."""
import numpy as np
from scipy.stats import norm

from oracle.nf4 import DELTA, nf4_codebook


def test_codebook_shape_order_and_ends():
    c = nf4_codebook()
    assert c.dtype == np.float32 and c.shape == (16,)
    assert np.all(np.diff(c) > 0)
    assert c[0] == -1.0 and c[7] == 0.0 and c[15] == 1.0


def test_codebook_values_are_normal_quantiles():
    c = nf4_codebook().astype(np.float64)
    pos = norm.ppf(0.5 + np.arange(1, 9) / 8.0 * (DELTA - 0.5))
    neg = norm.ppf(0.5 + np.arange(1, 8) / 7.0 * (DELTA - 0.5))
    expect = np.concatenate([-(neg / neg[-1])[::-1], [0.0], pos / pos[-1]])
    assert np.allclose(c, expect, rtol=0, atol=2e-7)


def test_codebook_committed_copy_matches():
    from tests.golden_io import GOLDEN
    import os
    vals = np.loadtxt(os.path.join(GOLDEN, "nf4_codebook.txt"), dtype=np.float64).astype(np.float32)
    assert np.array_equal(vals, nf4_codebook())
