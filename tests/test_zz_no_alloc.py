"""uq_gemm_noalloc (collected last on purpose): the GEMV entry point for callers that cannot let a
library allocate device memory -- runtimes that reserve all of it up front, or loops that cannot
afford the synchronisation an allocation implies.  Its scratch is a static device array inside the
library.  Through the C ABI this checks that two calls in a row (the second one finding the first
one's leftovers in that array) meet the oracle's pass rule and give exactly uq_gemm's bits (the same
kernel in the same order), that a split which needs the partial-sum area is covered, and that a
request too large for either part of the array is refused on its own."""
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
SCRATCH = 1 << 20


def _problem(fmt, group, M, N, K, seed):
    w = normal_weights(seed, N, K, 0.015 if fmt == "K4" else 0.02)
    x = activations(seed, M, K)
    qz = oquant.quantize(w, fmt, group, codebook=nf4_codebook() if fmt == "NF4" else None)
    wq, scales, zc = device_weights(qz, DEV)
    y_ref, b = ogemm.quantized_gemm(x, qz)
    return device_x(x, DEV), wq, scales, zc, y_ref, b


# (fmt, group, M, N, K, seed): whole row blocks per CTA, the stream-K split with its partial sums,
# the CUDA-core GEMV with tickets, two 8-row blocks of x
PROBLEMS = [("INT4_ASYM", 128, 1, 4104, 4096, 801), ("INT4_ASYM", 128, 3, 4096, 14336, 802),
            ("K4", 256, 8, 1024, 2304, 803), ("INT8_SYM", 128, 3, 1000, 1024, 804),
            ("NF4", 64, 12, 300, 1088, 805)]


def test_noalloc_matches_oracle_and_uq_gemm_on_two_calls_in_a_row():
    assert any(uq.gemm_kernel_count(M, N, K, g, f) == 2 for f, g, M, N, K, _ in PROBLEMS), \
        "no case takes the split that uses the partial-sum area"
    prepared = [(p, _problem(*p)) for p in PROBLEMS]
    ys = []
    for (fmt, group, M, N, K, _), (xd, wq, scales, zc, _, _) in prepared:
        y_gemm = uq.gemm(xd, wq, scales, zc, N, group, fmt)
        y_na = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        ys.append((y_gemm, y_na))
    torch.cuda.synchronize()
    for _ in range(2):   # the second round finds the first round's leftovers in the static array
        for ((fmt, group, M, N, K, _), (xd, wq, scales, zc, _, _)), (_, y_na) in zip(prepared, ys):
            y_na.fill_(float("nan"))
            uq.gemm_noalloc(xd, wq, scales, zc, N, group, fmt, y=y_na)
            torch.cuda.synchronize()
            assert uq.device_fault() == 0
        for ((fmt, group, M, N, K, _), (_, _, _, _, y_ref, b)), (y_gemm, y_na) in zip(prepared, ys):
            r = ogemm.error_ratio(y_to_f64(y_na), y_ref, b)
            assert np.isfinite(r).all() and r.max() <= 1.0, f"{fmt} {N}x{K} M={M}: max error ratio {r.max():.3g}"
            assert torch.equal(y_na.view(torch.int16), y_gemm.view(torch.int16)), f"{fmt}: differs from uq_gemm"


def _zeros_problem(N, K, group, fmt, M):
    wq_bytes, sc_bytes, z_bytes = uq.packed_size(N, K, group, fmt)
    xd = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
    wq = torch.zeros(wq_bytes, dtype=torch.uint8, device=DEV)
    sc = torch.zeros(sc_bytes // 2, dtype=torch.int16, device=DEV)
    zc = torch.zeros(max(z_bytes, 16), dtype=torch.uint8, device=DEV) if z_bytes else None
    y = torch.zeros((M, N), dtype=torch.bfloat16, device=DEV)
    return xd, wq, sc, zc, y


def test_noalloc_refuses_partial_sums_beyond_its_scratch():
    """4096 x 14336 INT4 at M = 8 takes the stream-K split: 256 row blocks x 14 k tiles x 16 rows x
    8 columns of fp32 partial sums (1.8 MB) exceed the array; this format uses no tickets."""
    N, K, group, fmt, M = 4096, 14336, 128, "INT4_ASYM", 8
    assert uq.gemm_kernel_count(M, N, K, group, fmt) == 2
    assert uq.gemm_noalloc_scratch(M, N, K, group, fmt) == (0, 256 * 14 * 16 * 8 * 4)
    assert 256 * 14 * 16 * 8 * 4 > SCRATCH
    xd, wq, sc, zc, y = _zeros_problem(N, K, group, fmt, M)
    with pytest.raises(uq.UqError) as e:
        uq.gemm_noalloc(xd, wq, sc, zc, N, group, fmt, y=y)
    assert e.value.status == 5
    # the same shape at M = 3 fits (256 * 14 * 16 * 3 * 4 bytes) and runs
    uq.gemm_noalloc(xd[:3].contiguous(), wq, sc, zc, N, group, fmt, y=y[:3].contiguous())
    torch.cuda.synchronize()
    assert uq.device_fault() == 0


def test_noalloc_needs_no_partial_sums_when_ctas_own_whole_row_blocks():
    """19456 x 4096 INT4_SYM at M = 8: every CTA owns whole 16-row blocks (one launch), so no scratch
    beyond the fault word is used, although the stream-K split of the same shape would need 2.5 MB of
    partial sums.  The output must equal uq_gemm's bit for bit."""
    N, K, group, fmt, M = 19456, 4096, 32, "INT4_SYM", 8
    assert uq.gemm_kernel_count(M, N, K, group, fmt) == 1
    assert uq.gemm_noalloc_scratch(M, N, K, group, fmt) == (0, 0)
    assert (N // 16) * (K // 1024) * 16 * M * 4 > SCRATCH
    g = torch.Generator(device=DEV)
    g.manual_seed(806)
    xd, wq, sc, zc, y = _zeros_problem(N, K, group, fmt, M)
    wq.copy_(torch.randint(0, 256, wq.shape, generator=g, device=DEV, dtype=torch.int32).to(torch.uint8))
    sc.copy_((torch.rand(sc.shape, generator=g, device=DEV) * 0.01).half().view(torch.int16))
    xd.copy_(torch.randn(xd.shape, generator=g, device=DEV).to(torch.bfloat16))
    y_gemm = uq.gemm(xd, wq, sc, zc, N, group, fmt)
    y.fill_(float("nan"))
    uq.gemm_noalloc(xd, wq, sc, zc, N, group, fmt, y=y)
    torch.cuda.synchronize()
    assert uq.device_fault() == 0
    assert torch.equal(y.view(torch.int16), y_gemm.view(torch.int16))
