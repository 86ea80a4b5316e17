"""GPU parity of the mma.sync GEMM against the oracle, every element.  uq_gemm routes 9..15 rows of the
4-bit and 2-bit formats and K4 at any M >= 9 to it; these tests select it for every M >= 9
(uq_set_gemm_path(2)) so that it is checked at every width: each format and group at M from 9 to 100 on a shape with a ragged
last row group and a narrower last k unit, the split of a long k range over several CTAs (second
pass), the 8-row GEMV tail of M = 70, determinism, and the gated projection's two passes.

Pass rule (oracle/gemm.py): |y - y_ref| <= 1e-3 * sum_k |x_k w_hat_k| + 1e-6.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import gemm_uq_gb300 as uq  # noqa: E402
from oracle import gemm as ogemm  # noqa: E402
from oracle import mlp as omlp  # noqa: E402
from oracle import quant as oquant  # noqa: E402
from synth import activations, normal_weights  # noqa: E402
from tests.uq_helpers import KT, device_weights, device_x, mma_gemm_launches, y_to_f64  # noqa: E402

DEV = torch.device("cuda:0")
FMTS = [("INT4_ASYM", 128), ("INT4_ASYM", 64), ("INT4_ASYM", 32), ("INT4_SYM", 32), ("INT4_SYM", 128),
        ("INT2_ASYM", 64), ("INT2_ASYM", 32), ("INT2_ASYM", 128), ("K4", 256)]


@pytest.fixture(autouse=True)
def _mma_gemm_path():
    uq.set_gemm_path("mma")
    yield
    uq.set_gemm_path("auto")
    assert uq.device_fault() == 0, "a kernel's bounded wait ran out"


def _case(fmt, group, M, N, K, seed):
    w = normal_weights(seed, N, K, 0.015 if fmt == "K4" else 0.02, outlier_p=0.001, outlier_mult=20.0)
    x = activations(seed, M, K)
    qz = oquant.quantize(w, fmt, group)
    wq, scales, zc = device_weights(qz, DEV)
    xd = device_x(x, DEV)
    y = uq.gemm(xd, wq, scales, zc, N, group, fmt)
    y_ref, b = ogemm.quantized_gemm(x, qz)
    return y, y_ref, b, (xd, wq, scales, zc)


@pytest.mark.parametrize("fmt,group", FMTS)
@pytest.mark.parametrize("M", [9, 16, 24, 33, 64])
def test_mma_gemm_parity(fmt, group, M):
    # 264 rows: two full 128-row groups and one of 8 rows; K: two full tiles and a narrower tail
    N, K = 264, 2 * KT[fmt] + (256 if fmt == "K4" else max(group, 64))
    y, y_ref, b, _ = _case(fmt, group, M, N, K, seed=1800 + M)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert np.isfinite(r).all() and r.max() <= 1.0, f"max error ratio {r.max():.3g}"


@pytest.mark.parametrize("M", [65, 70, 100])
def test_mma_gemm_beyond_64_rows(M):
    # blocks of 64 rows on the GEMM; 70 leaves a last block of 6 rows for the GEMV
    y, y_ref, b, _ = _case("INT4_ASYM", 128, M, 392, 3072, seed=1850 + M)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"


@pytest.mark.parametrize("fmt,group", [("INT4_ASYM", 128), ("K4", 256), ("INT2_ASYM", 64)])
def test_mma_gemm_split_k_range(fmt, group):
    """Few row groups, long K: each row group's k units are split over several CTAs, whose partial
    sums a second launch adds in split order."""
    N, K, M = 256, 16384, 24
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert uq.gemm_kernel_count(M, N, K, group, fmt) == mma_gemm_launches(fmt, N, K, sms)
    assert mma_gemm_launches(fmt, N, K, sms) >= (3 if fmt == "K4" else 2), "the shape must split its k range"
    y, y_ref, b, _ = _case(fmt, group, M, N, K, seed=1870)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"


@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_mma_gemm_full_size_every_row(N, K):
    y, y_ref, b, _ = _case("INT4_ASYM", 128, 64, N, K, seed=1880)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"


def test_mma_gemm_deterministic():
    y, _, _, (xd, wq, scales, zc) = _case("INT4_ASYM", 64, 40, 1024, 8192, seed=1890)
    for _ in range(3):
        y2 = uq.gemm(xd, wq, scales, zc, 1024, 64, "INT4_ASYM")
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_mma_gemm_and_tensor_cores_both_meet_the_rule():
    """The same call on the mma.sync GEMM and on the tcgen05 kernel (uq_set_gemm_path(1)): both within
    the rule; their rounding differs, so they are not compared bit for bit."""
    fmt, group, M, N, K = "INT4_ASYM", 128, 32, 512, 4096
    w = normal_weights(1895, N, K, 0.02)
    x = activations(1895, M, K)
    qz = oquant.quantize(w, fmt, group)
    wq, scales, zc = device_weights(qz, DEV)
    xd = device_x(x, DEV)
    y_ref, b = ogemm.quantized_gemm(x, qz)
    y_auto = uq.gemm(xd, wq, scales, zc, N, group, fmt)          # the mma.sync GEMM (this module's path)
    try:
        uq.set_gemm_path("tensor_cores")
        assert uq.gemm_kernel_count(M, N, K, group, fmt) == 1
        y_tc = uq.gemm(xd, wq, scales, zc, N, group, fmt)
    finally:
        uq.set_gemm_path("mma")
    for y in (y_auto, y_tc):
        assert ogemm.error_ratio(y_to_f64(y), y_ref, b).max() <= 1.0


def test_automatic_routing():
    """Automatic choice: the mma.sync GEMM for 9..15 rows and for K4, the tensor cores for wider INT4 blocks."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    uq.set_gemm_path("auto")
    try:
        assert uq.gemm_kernel_count(12, 14336, 4096, 128, "INT4_ASYM") == mma_gemm_launches("INT4_ASYM", 14336, 4096, sms)
        assert uq.gemm_kernel_count(32, 8192, 8192, 256, "K4") == mma_gemm_launches("K4", 8192, 8192, sms)
        assert uq.gemm_kernel_count(64, 14336, 4096, 128, "INT4_ASYM") == 1
    finally:
        uq.set_gemm_path("mma")


@pytest.mark.parametrize("M", [9, 16, 40])
def test_gated_on_the_mma_gemm(M):
    fmt, group, N, K = "INT4_ASYM", 128, 520, 2048
    wg = normal_weights(1900 + M, N, K, 0.02)
    wu = normal_weights(1950 + M, N, K, 0.02)
    x = activations(1990 + M, M, K)
    qg, qu = oquant.quantize(wg, fmt, group), oquant.quantize(wu, fmt, group)
    dg, du = device_weights(qg, DEV), device_weights(qu, DEV)
    h = uq.gemm_gated(device_x(x, DEV), dg, du, N, group, fmt)
    h_ref, bound = omlp.gated_quantized(x, qg, qu)
    r = omlp.gated_error_ratio(y_to_f64(h), h_ref, bound)
    assert np.isfinite(r).all() and r.max() <= 1.0, f"max error ratio {r.max():.3g}"
