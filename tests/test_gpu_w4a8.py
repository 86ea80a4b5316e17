"""GPU parity of W4A8 / W8A8 (uq_gemm_w4a8) against the oracle (oracle/w4a8.py), every element.

Pass rule: |y - y_ref| <= 1e-4 b' + 2^-8 |y_ref| + 1e-6, b' = s_x * sum_g |s_g| * sum_k |xq (q - z)|.
The activation codes are taken in fp32 on both sides, so the integer sums agree exactly and only the
fp32 scaling and the bf16 output rounding remain.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import gemm_uq_gb300 as uq  # noqa: E402
from oracle import quant as oquant  # noqa: E402
from oracle import w4a8 as ow4a8  # noqa: E402
from synth import activations, normal_weights  # noqa: E402
from tests.uq_helpers import KT, device_weights, device_x, y_to_f64  # noqa: E402

DEV = torch.device("cuda:0")
FMTS = [("INT4_SYM", 32), ("INT4_ASYM", 128), ("INT4_ASYM", 64), ("INT8_SYM", 128), ("INT8_SYM", 32)]


@pytest.fixture(autouse=True)
def _no_fault():
    yield
    assert uq.device_fault() == 0


def _case(fmt, group, M, N, K, seed, zero_row=False):
    w = normal_weights(seed, N, K, 0.02, outlier_p=0.001, outlier_mult=20.0)
    x = activations(seed, M, K)
    if zero_row and M > 1:
        x[1] = 0.0
    qz = oquant.quantize(w, fmt, group)
    wq, scales, zc = device_weights(qz, DEV)
    y = uq.gemm_w4a8(device_x(x, DEV), wq, scales, zc, N, group, fmt)
    y_ref, b = ow4a8.w4a8_reference(x, qz)
    return y, y_ref, b, (x, wq, scales, zc)


@pytest.mark.parametrize("fmt,group", FMTS)
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_w4a8_parity_small(fmt, group, M):
    N, K = 300, 2 * KT[fmt] + 128
    y, y_ref, b, _ = _case(fmt, group, M, N, K, seed=1500 + M, zero_row=True)
    r = ow4a8.error_ratio(y_to_f64(y), y_ref, b)
    assert np.isfinite(r).all() and r.max() <= 1.0, f"max error ratio {r.max():.3g}"
    if M > 1:
        assert torch.count_nonzero(y[1].float()) == 0                  # the zero row of x


@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_w4a8_full_size_every_row(N, K):
    fmt, group = "INT4_ASYM", 128
    y, y_ref, b, _ = _case(fmt, group, 1, N, K, seed=1600)
    r = ow4a8.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"


def test_w4a8_deterministic_and_kernel_count():
    fmt, group = "INT4_ASYM", 128
    y, _, _, (x, wq, scales, zc) = _case(fmt, group, 4, 1024, 4096, seed=1700)
    y2 = uq.gemm_w4a8(device_x(x, DEV), wq, scales, zc, 1024, group, fmt)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert uq.gemm_w4a8_kernel_count(1, 14336, 4096, 128, "INT4_ASYM") == 2     # x codes + one GEMV launch
    # 4096 x 14336: whole row blocks per CTA (x codes fit beside the ring), no second pass; at 8 rows
    # the stream-K split and its second pass
    assert uq.gemm_w4a8_kernel_count(1, 4096, 14336, 128, "INT4_ASYM") == 2
    assert uq.gemm_w4a8_kernel_count(8, 4096, 14336, 128, "INT4_ASYM") == 3
    with pytest.raises(uq.UqError):
        uq.gemm_w4a8_kernel_count(1, 64, 256, 64, "NF4")


@pytest.mark.parametrize("fmt,group", [("INT4_ASYM", 128), ("INT8_SYM", 128), ("INT4_SYM", 32)])
def test_w4a8_rows_alone_and_batched(fmt, group):
    # the integer sums are exact and the fp32 folds run in the same order for any M, so every row of
    # a batch equals the row alone bit for bit (ragged last tile and row block included)
    N, K, M = 300, 2 * KT[fmt] + 128, 8
    y, _, _, (x, wq, scales, zc) = _case(fmt, group, M, N, K, seed=1800)
    xd = device_x(x, DEV)
    for m in range(M):
        y1 = uq.gemm_w4a8(xd[m:m + 1].contiguous(), wq, scales, zc, N, group, fmt)
        assert torch.equal(y1[0].view(torch.int16), y[m].view(torch.int16)), f"row {m} differs from M=1 call"
