"""GGUF Q4_0 / Q8_0 blocks through the library: uq_pack_gguf, then the kernels of the group-32 symmetric
formats.  Codes and W_hat bit-exact against the oracle's block decoder; y within the linear layers' pass
rule on the GEMV and tensor-core paths, every element, including a full 8192 x 8192 weight."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import gemm_uq_gb300 as uq  # noqa: E402
from oracle import gemm as ogemm  # noqa: E402
from oracle import gguf as ogguf  # noqa: E402
from synth import activations, gguf_blocks  # noqa: E402
from tests.uq_helpers import device_x, y_to_f64  # noqa: E402

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _no_fault():
    yield
    assert uq.device_fault() == 0


@pytest.mark.parametrize("qtype", ["Q4_0", "Q8_0"])
@pytest.mark.parametrize("N,K", [(300, 2048 + 64), (37, 32), (128, 4096)])
def test_gguf_codes_and_dequant_bit_exact(qtype, N, K):
    raw = gguf_blocks(1200 + N, N, K, qtype)
    wq, scales = uq.pack_gguf(torch.from_numpy(raw).to(DEV), qtype, N, K)
    fmt = uq.GGUF_TYPES[qtype][1]
    _, codes = ogguf.split_blocks(raw, qtype, N, K)
    assert np.array_equal(uq.unpack_codes(wq, N, K, 32, fmt).cpu().numpy(), codes)
    got = uq.dequant(wq, scales, None, N, K, 32, fmt).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ogguf.dequant(raw, qtype, N, K).view(np.uint32))


@pytest.mark.parametrize("qtype", ["Q4_0", "Q8_0"])
@pytest.mark.parametrize("M", [1, 3, 8, 16, 40])
def test_gguf_gemm_parity(qtype, M):
    N, K = 264, 2048
    raw = gguf_blocks(1300 + M, N, K, qtype)
    wq, scales = uq.pack_gguf(torch.from_numpy(raw).to(DEV), qtype, N, K)
    x = activations(1301 + M, M, K)
    y = uq.gemm(device_x(x, DEV), wq, scales, None, N, 32, uq.GGUF_TYPES[qtype][1])
    y_ref, b = ogemm.reference(x, ogguf.dequant(raw, qtype, N, K))
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"


@pytest.mark.parametrize("qtype", ["Q4_0", "Q8_0"])
def test_gguf_full_size_every_row(qtype):
    N = K = 8192
    raw = gguf_blocks(1400, N, K, qtype)
    wq, scales = uq.pack_gguf(torch.from_numpy(raw).to(DEV), qtype, N, K)
    w_hat = ogguf.dequant(raw, qtype, N, K)
    for M in (1, 16):
        x = activations(1401 + M, M, K)
        y = uq.gemm(device_x(x, DEV), wq, scales, None, N, 32, uq.GGUF_TYPES[qtype][1])
        y_ref, b = ogemm.reference(x, w_hat)
        r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
        assert r.max() <= 1.0, f"{qtype} M={M}: max error ratio {r.max():.3g}"


def test_gguf_rejects_unaligned_k():
    raw = torch.zeros(100, dtype=torch.uint8, device=DEV)
    with pytest.raises(uq.UqError):
        uq.pack_gguf(raw, "Q4_0", 2, 48)
