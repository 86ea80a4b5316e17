"""uq_gemm_noalloc (collected last on purpose): the GEMV entry point for callers that cannot let a
library allocate device memory -- runtimes that reserve all of it up front, or loops that cannot
afford the synchronisation an allocation implies.  Its scratch is a static device array inside the
library; this checks, through the C ABI, that two calls in a row (the second one finding the first
one's leftovers in that array) give what uq_gemm gives, within the pass rule the other tests use."""
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


def _problem(fmt, group, M, N, K, seed):
    w = normal_weights(seed, N, K, 0.015 if fmt == "K4" else 0.02)
    x = activations(seed, M, K)
    qz = oquant.quantize(w, fmt, group, codebook=nf4_codebook() if fmt == "NF4" else None)
    wq, scales, zc = device_weights(qz, DEV)
    _, b = ogemm.quantized_gemm(x, qz)
    return device_x(x, DEV), wq, scales, zc, b


def test_noalloc_matches_uq_gemm_on_two_calls_in_a_row():
    problems = [("INT4_ASYM", 128, 1, 4104, 4096, 801), ("K4", 256, 8, 1024, 2304, 802)]
    prepared = [(p, _problem(*p)) for p in problems]
    outs = []
    for (fmt, group, M, N, K, _), (xd, wq, scales, zc, b) in prepared:
        y_ref = uq.gemm(xd, wq, scales, zc, N, group, fmt)
        y_na = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        outs.append((fmt, y_ref, y_na, b))
    # the two no-alloc calls back to back on the same stream
    for ((fmt, group, M, N, K, _), (xd, wq, scales, zc, b)), (_, _, y_na, _) in zip(prepared, outs):
        uq.gemm_noalloc(xd, wq, scales, zc, N, group, fmt, y=y_na)
    torch.cuda.synchronize()
    assert uq.device_fault() == 0
    for fmt, y_ref, y_na, b in outs:
        r = ogemm.error_ratio(y_to_f64(y_na), y_to_f64(y_ref), b)
        assert np.isfinite(r).all() and r.max() <= 1.0, f"{fmt}: max error ratio {r.max():.3g}"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    """N one row block past the static ticket area.  Every buffer is sized for the request, so
    the call would only read valid memory even if the size check did not fire."""
    N, K, group, fmt = 1048576 + 16, 32, 32, "INT4_SYM"
    wq_bytes, sc_bytes, _ = uq.packed_size(N, K, group, fmt)
    xd = torch.zeros((1, K), dtype=torch.bfloat16, device=DEV)
    wq = torch.zeros(wq_bytes, dtype=torch.uint8, device=DEV)
    sc = torch.zeros(sc_bytes // 2, dtype=torch.int16, device=DEV)
    y = torch.zeros((1, N), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(uq.UqError) as e:
        uq.gemm_noalloc(xd, wq, sc, None, N, group, fmt, y=y)
    assert e.value.status == 5
