"""GPU parity of the gated projection h = silu(x Wg^T) * (x Wu^T) (uq_gemm_gated) against the oracle.

Pass rule (oracle/mlp.py): |h - h_ref| <= 1e-3 * (1.1 b_g |u| + |silu(g)| b_u) + 2^-8 |h_ref| + 1e-6.
Small ragged shapes cover every format on the GEMV (M <= 15) and tensor-core (M >= 16) paths; the
full-size cases compare every output element of the 8B and 70B gate/up shapes.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import gemm_uq_gb300 as uq  # noqa: E402
from oracle import mlp as omlp  # noqa: E402
from oracle import quant as oquant  # noqa: E402
from oracle.nf4 import nf4_codebook  # noqa: E402
from synth import activations, normal_weights  # noqa: E402
from tests.uq_helpers import mma_gemm_launches, KT, device_weights, device_x, y_to_f64  # noqa: E402

DEV = torch.device("cuda:0")
FMT_GROUPS = [("INT4_SYM", 32), ("INT4_ASYM", 128), ("INT8_SYM", 128), ("INT2_ASYM", 64), ("NF4", 64), ("K4", 256)]


@pytest.fixture(autouse=True)
def _no_fault():
    yield
    assert uq.device_fault() == 0, "a kernel's bounded wait ran out"


def _quantize(w, fmt, group):
    if fmt == "K4":
        return oquant.quantize_k4(w)
    return oquant.quantize(w, fmt, group, codebook=nf4_codebook() if fmt == "NF4" else None)


def _case(fmt, group, M, N, K, seed):
    sigma = 0.015 if fmt == "K4" else 0.02
    wg = normal_weights(seed, N, K, sigma, outlier_p=0.001, outlier_mult=20.0)
    wu = normal_weights(seed + 1, N, K, sigma, outlier_p=0.001, outlier_mult=20.0)
    x = activations(seed, M, K)
    qg, qu = _quantize(wg, fmt, group), _quantize(wu, fmt, group)
    gate, up = device_weights(qg, DEV), device_weights(qu, DEV)
    h = uq.gemm_gated(device_x(x, DEV), gate, up, N, group, fmt)
    h_ref, B = omlp.gated_quantized(x, qg, qu)
    return h, h_ref, B, (x, gate, up)


@pytest.mark.parametrize("fmt,group", FMT_GROUPS)
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16, 33])
def test_gated_parity_small(fmt, group, M):
    N, K = 300, 2 * KT[fmt] + (256 if fmt == "K4" else 128)
    h, h_ref, B, _ = _case(fmt, group, M, N, K, seed=600 + M)
    r = omlp.gated_error_ratio(y_to_f64(h), h_ref, B)
    assert np.isfinite(r).all() and r.max() <= 1.0, f"max error ratio {r.max():.3g}"


@pytest.mark.parametrize("fmt,group,M", [("INT4_ASYM", 128, 1), ("INT4_ASYM", 128, 8), ("K4", 256, 32)])
def test_gated_deterministic(fmt, group, M):
    N, K = 300, 2048
    h, _, _, (x, gate, up) = _case(fmt, group, M, N, K, seed=650)
    h2 = uq.gemm_gated(device_x(x, DEV), gate, up, N, group, fmt)
    assert torch.equal(h.view(torch.int16), h2.view(torch.int16))


def test_gated_edge_cases():
    fmt, group = "INT4_ASYM", 128
    h = torch.full((2, 5), 7.0, dtype=torch.bfloat16, device=DEV)
    x = torch.zeros((2, 0), dtype=torch.bfloat16, device=DEV)
    dummy = torch.zeros(16, dtype=torch.uint8, device=DEV)
    uq.gemm_gated(x, (dummy, dummy, dummy), (dummy, dummy, dummy), 5, group, fmt, h=h)
    assert torch.count_nonzero(h.float()) == 0
    # a zero up projection gives exact zeros whatever the gate
    N, K = 48, 256
    wg = normal_weights(660, N, K, 0.02)
    qg = oquant.quantize(wg, fmt, group)
    qz = oquant.quantize(np.zeros((N, K), np.float32), fmt, group)
    hz = uq.gemm_gated(device_x(activations(661, 3, K), DEV), device_weights(qg, DEV), device_weights(qz, DEV),
                       N, group, fmt)
    assert torch.count_nonzero(hz.float()) == 0


def test_gated_kernel_count():
    # decode (mma GEMV formats, M <= 8): gate and up in one launch, plus the second pass when the work
    # split shares row blocks; the mma.sync GEMM (M >= 9), INT8 / NF4 and the tensor-core path: a
    # gate pass and an up pass
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    gemm = mma_gemm_launches("INT4_ASYM", 14336, 4096, sms)
    assert uq.gemm_gated_kernel_count(1, 14336, 4096, 128, "INT4_ASYM") == 1
    assert uq.gemm_gated_kernel_count(1, 28672, 8192, 256, "K4") == 2
    assert uq.gemm_gated_kernel_count(9, 14336, 4096, 128, "INT4_ASYM") == 2 * gemm
    assert uq.gemm_gated_kernel_count(1, 8192, 8192, 128, "INT8_SYM") == 2
    assert uq.gemm_gated_kernel_count(16, 14336, 4096, 128, "INT4_ASYM") == 2               # tensor cores
    assert uq.gemm_gated_kernel_count(70, 14336, 4096, 128, "INT4_ASYM") == 4               # two 64-row blocks
    assert uq.gemm_gated_kernel_count(0, 14336, 4096, 128, "INT4_ASYM") == 0


@pytest.mark.parametrize("fmt,group,N,K,Ms", [("INT4_ASYM", 128, 14336, 4096, [1, 8, 16, 64]),
                                              ("K4", 256, 28672, 8192, [1, 32])])
def test_gated_full_size_every_row(fmt, group, N, K, Ms):
    """The 8B-shaped (14336 x 4096) and 70B-shaped (28672 x 8192) gate/up pairs, every output element."""
    sigma = 0.015 if fmt == "K4" else 0.02
    wg = normal_weights(670, N, K, sigma, outlier_p=0.001, outlier_mult=20.0)
    wu = normal_weights(671, N, K, sigma, outlier_p=0.001, outlier_mult=20.0)
    rows = 2048
    q = {}
    for name, w in (("g", wg), ("u", wu)):
        parts = [_quantize(w[r0:r0 + rows], fmt, group) for r0 in range(0, N, rows)]
        q[name] = parts
    # device weights: the oracle's codes and metadata, packed by the library
    def dev_of(parts):
        whole = oquant.Quantized(fmt, group, np.concatenate([p.codes for p in parts]))
        if fmt == "K4":
            for f in ("d", "dmin", "sc", "m"):
                setattr(whole, f, np.concatenate([getattr(p, f) for p in parts]))
        else:
            whole.scale = np.concatenate([p.scale for p in parts])
            whole.zero = np.concatenate([p.zero for p in parts]) if parts[0].zero is not None else None
        return device_weights(whole, DEV)
    gate, up = dev_of(q["g"]), dev_of(q["u"])
    for M in Ms:
        x = activations(672 + M, M, K)
        h = y_to_f64(uq.gemm_gated(device_x(x, DEV), gate, up, N, group, fmt))
        worst = 0.0
        for i, r0 in enumerate(range(0, N, rows)):
            h_ref, B = omlp.gated_quantized(x, q["g"][i], q["u"][i])
            worst = max(worst, float(omlp.gated_error_ratio(h[:, r0:r0 + rows], h_ref, B).max()))
        assert worst <= 1.0, f"{fmt} {N}x{K} M={M}: max error ratio {worst:.3g}"
