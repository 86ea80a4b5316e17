"""GPU parity of the tcgen05 tensor-core path (M >= 16): shapes it serves (N % 8 == 0, K a multiple of
the code tile width), including a ragged last 128-row block and M that is not a multiple of 16.  Every
test here selects the tensor-core path for all formats (uq_set_gemm_path(1)); by default the 4-bit and
2-bit formats take the mma.sync GEMM instead (tests/test_gpu_gemm_mma.py)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import gemm_uq_gb300 as uq  # noqa: E402
from oracle import gemm as ogemm  # noqa: E402
from oracle import quant as oquant  # noqa: E402
from oracle.nf4 import nf4_codebook  # noqa: E402
from synth import activations, normal_weights  # noqa: E402
from tests.uq_helpers import device_weights, device_x, y_to_f64  # noqa: E402

DEV = torch.device("cuda:0")
TC_FMTS = [("INT4_ASYM", 128), ("INT4_ASYM", 32), ("INT4_SYM", 32), ("INT4_SYM", 128), ("INT8_SYM", 128),
           ("INT8_SYM", 32), ("K4", 256), ("INT2_ASYM", 64), ("INT2_ASYM", 32), ("INT2_ASYM", 128), ("NF4", 64),
           ("NF4", 32), ("NF4", 128)]


@pytest.fixture(autouse=True)
def _tensor_core_path():
    uq.set_gemm_path("tensor_cores")
    yield
    uq.set_gemm_path("auto")
    assert uq.device_fault() == 0, "a kernel's bounded wait ran out"


def _case(fmt, group, M, N, K, seed):
    w = normal_weights(seed, N, K, 0.015 if fmt == "K4" else 0.02, outlier_p=0.001, outlier_mult=20.0)
    x = activations(seed, M, K)
    qz = oquant.quantize(w, fmt, group, codebook=nf4_codebook() if fmt == "NF4" else None)
    wq, scales, zc = device_weights(qz, DEV)
    xd = device_x(x, DEV)
    y = uq.gemm(xd, wq, scales, zc, N, group, fmt)
    y_ref, b = ogemm.quantized_gemm(x, qz)
    return y, y_ref, b, (xd, wq, scales, zc)


def test_tc_smoke_small():
    """One small tensor-core call first: a single 128-row block, one k tile, M = 16."""
    y, y_ref, b, _ = _case("INT4_ASYM", 128, 16, 128, 1024, seed=600)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"


@pytest.mark.parametrize("fmt,group", TC_FMTS)
@pytest.mark.parametrize("M", [16, 17, 32, 48, 64])
def test_tc_parity(fmt, group, M):
    N, K = 264, 2048                      # two full 128-row blocks + a ragged one of 8 rows
    y, y_ref, b, _ = _case(fmt, group, M, N, K, seed=610 + M)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"


@pytest.mark.parametrize("M", [65, 100, 130])
def test_tc_parity_wide_m(M):
    y, y_ref, b, _ = _case("INT4_ASYM", 128, M, 384, 3072, seed=650 + M)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"


def test_tc_serves_every_format_in_one_launch():
    """M >= 16 with K a multiple of the code tile: one tensor-core launch for every format (K4: after its
    x column-sum pre-kernel), no 8-row GEMV blocks."""
    for fmt, group in [("INT4_SYM", 32), ("INT4_ASYM", 128), ("INT8_SYM", 128), ("INT2_ASYM", 64), ("NF4", 64)]:
        assert uq.gemm_kernel_count(16, 8192, 8192, group, fmt) == 1, fmt
    assert uq.gemm_kernel_count(16, 8192, 8192, 256, "K4") == 2


@pytest.mark.parametrize("fmt,group", [("INT4_ASYM", 128), ("K4", 256), ("INT2_ASYM", 64), ("NF4", 64)])
def test_tc_deterministic(fmt, group):
    y, _, _, (xd, wq, scales, zc) = _case(fmt, group, 32, 1024, 4096, seed=700)
    for _ in range(3):
        y2 = uq.gemm(xd, wq, scales, zc, 1024, group, fmt)
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_tc_split_row_blocks_many_ctas():
    """Few row blocks, long K: every 128-row block is split over several CTAs (ticketed reduction)."""
    y, y_ref, b, _ = _case("INT4_ASYM", 128, 16, 256, 16384, seed=710)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"
