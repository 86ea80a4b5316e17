"""GPU: uq_set_launch_overlap (programmatic dependent launch) keeps chained calls correct --
the second linear reads the first one's output as its x, on the same stream, eagerly and inside a
captured CUDA graph -- and gives bit-identical results to the plain launches."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import gemm_uq_gb300 as uq  # noqa: E402
from oracle import quant as oquant  # noqa: E402
from synth import activations, normal_weights  # noqa: E402
from tests.uq_helpers import device_weights, device_x  # noqa: E402

DEV = torch.device("cuda:0")


def _layer(seed, N, K):
    qz = oquant.quantize(normal_weights(seed, N, K, 0.02), "INT4_ASYM", 128)
    return device_weights(qz, DEV)


def _chain(layers, x, M, reps):
    outs = []
    for _ in range(reps):
        h = x
        for (wq, sc, zc), N in layers:
            h = uq.gemm(h, wq, sc, zc, N, 128, "INT4_ASYM")
        outs.append(h)
    return outs


@pytest.mark.parametrize("M", [1, 5, 16, 33])
def test_overlap_chain_matches_plain(M):
    # K of every layer a multiple of 1024, so M >= 16 runs the tensor-core path
    dims = [4096, 2048, 4096, 3072, 4096]
    layers = [(_layer(900 + i, dims[i + 1], dims[i]), dims[i + 1]) for i in range(len(dims) - 1)]
    x = device_x(activations(901, M, dims[0]), DEV)
    try:
        uq.set_launch_overlap(False)
        ref = _chain(layers, x, M, 3)
        torch.cuda.synchronize()
        uq.set_launch_overlap(True)
        got = _chain(layers, x, M, 3)
        torch.cuda.synchronize()
        for r, g in zip(ref, got):
            assert torch.equal(r.view(torch.int16), g.view(torch.int16))
        # the same chain captured in a graph and replayed
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            _chain(layers, x, M, 1)          # workspace for this stream, outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            out = _chain(layers, x, M, 1)[0]
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref[0].view(torch.int16))
    finally:
        uq.set_launch_overlap(False)
    assert uq.device_fault() == 0
