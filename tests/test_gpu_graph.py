"""A CUDA graph captured before the library's workspace grows stays valid after the growth.

uq_gemm keeps split-K partial sums in a per-(device, stream) workspace that a larger call grows.  A
graph captured earlier holds the old buffer's address; the library keeps replaced buffers allocated
until exit, so replaying that graph after an eager call that grew the workspace must still give the
oracle's result (and the same bits as before the growth).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import gemm_uq_gb300 as uq  # noqa: E402
from oracle import gemm as ogemm  # noqa: E402
from oracle import quant as oquant  # noqa: E402
from synth import activations, normal_weights  # noqa: E402
from tests.uq_helpers import device_weights, device_x, y_to_f64  # noqa: E402

DEV = torch.device("cuda:0")


def _case(N, K, M, seed):
    w = normal_weights(seed, N, K, 0.02)
    x = activations(seed, M, K)
    qz = oquant.quantize(w, "INT4_ASYM", 128)
    wq, scales, zc = device_weights(qz, DEV)
    y_ref, b = ogemm.quantized_gemm(x, qz)
    return device_x(x, DEV), wq, scales, zc, y_ref, b


def test_graph_replay_after_workspace_growth():
    # small: 1024 x 14336 at M = 1 splits row blocks between CTAs (partial sums in the workspace);
    # large: 4096 x 14336 at M = 4 needs a larger workspace
    small = uq.gemm_noalloc_scratch(1, 1024, 14336, 128, "INT4_ASYM")[1]
    large = uq.gemm_noalloc_scratch(4, 4096, 14336, 128, "INT4_ASYM")[1]
    assert 0 < small < large
    xs, wqs, ss, zs, y_ref_s, b_s = _case(1024, 14336, 1, 901)
    xl, wql, sl, zl, y_ref_l, b_l = _case(4096, 14336, 4, 902)
    st = torch.cuda.Stream(device=DEV)
    ys = torch.empty((1, 1024), dtype=torch.bfloat16, device=DEV)
    with torch.cuda.stream(st):
        uq.gemm(xs, wqs, ss, zs, 1024, 128, "INT4_ASYM", y=ys)      # sizes this stream's workspace
    st.synchronize()
    y_eager = ys.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        uq.gemm(xs, wqs, ss, zs, 1024, 128, "INT4_ASYM", y=ys)
    with torch.cuda.stream(st):
        yl = uq.gemm(xl, wql, sl, zl, 4096, 128, "INT4_ASYM")       # grows the workspace
    st.synchronize()
    ys.fill_(float("nan"))
    for _ in range(3):
        with torch.cuda.stream(st):
            g.replay()
    st.synchronize()
    assert uq.device_fault() == 0
    assert torch.equal(ys.view(torch.int16), y_eager.view(torch.int16))
    r = ogemm.error_ratio(y_to_f64(ys), y_ref_s, b_s)
    assert np.isfinite(r).all() and r.max() <= 1.0
    r = ogemm.error_ratio(y_to_f64(yl), y_ref_l, b_l)
    assert r.max() <= 1.0
