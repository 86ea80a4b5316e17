"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element.

Bit-exact: packed/unpacked codes, dequantized fp32 weights, the GPU quantizer's codes and
metadata.  Tolerance (the stated pass rule): |y - y_ref| <= 1e-3 * sum_k |x * w_hat| + 1e-6.
Shapes span several tiles with ragged row blocks (N % 8 != 0) and ragged k tiles.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import gemm_uq_gb300 as uq  # noqa: E402
from oracle import gemm as ogemm  # noqa: E402
from oracle import quant as oquant  # noqa: E402
from oracle.nf4 import nf4_codebook  # noqa: E402
from synth import activations, normal_weights  # noqa: E402
from tests.uq_helpers import KT, device_weights, device_x, h16, y_to_f64  # noqa: E402

DEV = torch.device("cuda:0")
FMT_GROUPS = [("INT4_SYM", 32), ("INT4_ASYM", 128), ("INT8_SYM", 128), ("INT2_ASYM", 64), ("NF4", 64),
              ("K4", 256), ("INT4_ASYM", 32), ("INT2_ASYM", 32), ("INT4_SYM", 128), ("NF4", 128)]
RANGES = {"INT4_SYM": (-8, 7), "INT4_ASYM": (0, 15), "INT8_SYM": (-128, 127), "INT2_ASYM": (0, 3),
          "NF4": (0, 15), "K4": (0, 15)}


def _k_ragged(fmt, group):
    """K spanning two full k tiles plus a narrower last one."""
    tail = max(group, 256 if fmt == "K4" else 64)
    return 2 * KT[fmt] + tail


def _quantize(w, fmt, group):
    return oquant.quantize(w, fmt, group, codebook=nf4_codebook() if fmt == "NF4" else None)


@pytest.fixture(autouse=True)
def _no_fault():
    yield
    assert uq.device_fault() == 0, "a kernel's bounded wait ran out"


@pytest.mark.parametrize("fmt,group", FMT_GROUPS)
def test_pack_unpack_bit_exact(fmt, group):
    N, K = 37, _k_ragged(fmt, group)
    lo, hi = RANGES[fmt]
    codes = np.random.default_rng(1).integers(lo, hi + 1, (N, K)).astype(np.int8)
    wq = uq.pack_layout(torch.from_numpy(codes).to(DEV), group, fmt)
    back = uq.unpack_codes(wq, N, K, group, fmt).cpu().numpy()
    assert np.array_equal(back, codes)


@pytest.mark.parametrize("fmt", ["INT4_SYM", "INT4_ASYM", "INT2_ASYM", "K4"])
def test_pack_rejects_out_of_range(fmt):
    group = 256 if fmt == "K4" else 64
    codes = np.zeros((8, 256), dtype=np.int8)
    codes[3, 17] = RANGES[fmt][1] + 1
    with pytest.raises(uq.UqError) as e:
        uq.pack_layout(torch.from_numpy(codes).to(DEV), group, fmt)
    assert e.value.status == 1


@pytest.mark.parametrize("fmt,group", FMT_GROUPS)
def test_dequant_bit_exact(fmt, group):
    N, K = 37, _k_ragged(fmt, group)
    w = normal_weights(31, N, K, 0.02, outlier_p=0.002, outlier_mult=20.0)
    qz = _quantize(w, fmt, group)
    wq, scales, zc = device_weights(qz, DEV)
    got = uq.dequant(wq, scales, zc, N, K, group, fmt).cpu().numpy()
    want = oquant.dequant(qz)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("fmt,group", [fg for fg in FMT_GROUPS if fg[0] != "K4"])
def test_gpu_quantizer_bit_exact(fmt, group):
    N, K = 37, 4 * 256
    w = normal_weights(32, N, K, 0.02, outlier_p=0.002, outlier_mult=20.0)
    w[3, :group] = 0.0                      # an all-zero group
    qz = _quantize(w, fmt, group)
    cb = torch.from_numpy(qz.codebook).to(DEV) if fmt == "NF4" else None
    codes, scales, zeros = uq.quantize(torch.from_numpy(w).to(DEV), group, fmt, codebook=cb)
    assert np.array_equal(codes.cpu().numpy(), qz.codes)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), qz.scale.view(np.uint16))
    if fmt == "INT4_ASYM":
        assert np.array_equal(zeros.cpu().numpy(), qz.zero)
        packed = uq.pack_zeros(zeros).cpu().numpy()
        assert np.array_equal(packed, oquant.pack_zero_nibbles(qz.zero))
    if fmt == "INT2_ASYM":
        assert np.array_equal(zeros.cpu().numpy().view(np.uint16), qz.zero.view(np.uint16))


def test_gpu_k4_quantizer_bit_exact():
    N, K = 21, 1024
    w = normal_weights(33, N, K, 0.015)
    w[2, :256] = np.abs(w[2, :256])         # a super-block with no negative weight (dmin = 0)
    w[4, 256:512] = 0.0                     # an all-zero super-block
    qz = oquant.quantize_k4(w)
    codes, d, dmin, sc, m = uq.quantize_k4(torch.from_numpy(w).to(DEV))
    assert np.array_equal(codes.cpu().numpy(), qz.codes)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), qz.d.view(np.uint16))
    assert np.array_equal(dmin.cpu().numpy().view(np.uint16), qz.dmin.view(np.uint16))
    assert np.array_equal(sc.cpu().numpy(), qz.sc)
    assert np.array_equal(m.cpu().numpy(), qz.m)


def _gemm_case(fmt, group, M, N, K, seed):
    w = normal_weights(seed, N, K, 0.015 if fmt == "K4" else 0.02, outlier_p=0.001, outlier_mult=20.0)
    x = activations(seed, M, K)
    qz = _quantize(w, fmt, group)
    wq, scales, zc = device_weights(qz, DEV)
    y = uq.gemm(device_x(x, DEV), wq, scales, zc, N, group, fmt)
    y_ref, b = ogemm.quantized_gemm(x, qz)
    return y, y_ref, b, (x, wq, scales, zc)


@pytest.mark.parametrize("fmt,group", FMT_GROUPS)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16])
def test_gemm_parity_small(fmt, group, M):
    N, K = 300, _k_ragged(fmt, group)
    y, y_ref, b, _ = _gemm_case(fmt, group, M, N, K, seed=40 + M)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"


@pytest.mark.parametrize("M", [17, 33, 64])
def test_gemm_parity_larger_m(M):
    N, K = 300, 2048 + 128
    y, y_ref, b, _ = _gemm_case("INT4_ASYM", 128, M, N, K, seed=70 + M)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"


def test_tiny_int4_workload_exact_config():
    """The tiny INT4 GEMV: M=1, N=K=256, symmetric INT4, group 32, N(0, 0.02), seed 0."""
    w = normal_weights(0, 256, 256, 0.02)
    x = activations(0, 1, 256)
    qz = oquant.quantize(w, "INT4_SYM", 32)
    wq, scales, zc = device_weights(qz, DEV)
    y = uq.gemm(device_x(x, DEV), wq, scales, zc, 256, 32, "INT4_SYM")
    y_ref, b = ogemm.quantized_gemm(x, qz)
    assert ogemm.error_ratio(y_to_f64(y), y_ref, b).max() <= 1.0


@pytest.mark.parametrize("fmt,group", [("INT4_ASYM", 128), ("NF4", 64), ("K4", 256), ("INT8_SYM", 128)])
def test_determinism_and_batched_rows(fmt, group):
    N, K, M = 300, _k_ragged(fmt, group), 8
    y, _, _, (x, wq, scales, zc) = _gemm_case(fmt, group, M, N, K, seed=90)
    xd = device_x(x, DEV)
    y2 = uq.gemm(xd, wq, scales, zc, N, group, fmt)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "repeat run not bit-identical"
    for m in range(M):
        y1 = uq.gemm(xd[m:m + 1].contiguous(), wq, scales, zc, N, group, fmt)
        assert torch.equal(y1[0].view(torch.int16), y[m].view(torch.int16)), f"row {m} differs from M=1 call"


def test_kernel_count_matches_the_paths():
    # 14336 x 4096 at M = 1: whole row blocks per CTA, one launch; 4096 x 14336: the stream-K split
    # and its second pass; the tensor-core path: one GEMM per 64 rows (K4: after its x column-sum
    # pre-kernel); M = 20 on the GEMV formats without tensor cores: three 8-row blocks
    assert uq.gemm_kernel_count(1, 14336, 4096, 128, "INT4_ASYM") == 1
    assert uq.gemm_kernel_count(1, 4096, 14336, 128, "INT4_ASYM") == 2
    assert uq.gemm_kernel_count(1, 8192, 8192, 128, "INT8_SYM") == 1
    assert uq.gemm_kernel_count(64, 14336, 4096, 128, "INT4_ASYM") == 1
    assert uq.gemm_kernel_count(128, 14336, 4096, 128, "INT4_ASYM") == 2
    assert uq.gemm_kernel_count(32, 8192, 8192, 256, "K4") == 2
    assert uq.gemm_kernel_count(20, 4096, 4096, 64, "NF4") == 3


def test_edge_cases():
    fmt, group = "INT4_ASYM", 128
    # M == 0 and N == 0 are no-ops; K == 0 writes zeros
    y = torch.full((2, 5), 7.0, dtype=torch.bfloat16, device=DEV)
    x = torch.zeros((2, 0), dtype=torch.bfloat16, device=DEV)
    dummy = torch.zeros(16, dtype=torch.uint8, device=DEV)
    uq.gemm(x, dummy, dummy, dummy, 5, group, fmt, y=y)
    assert torch.count_nonzero(y.float()) == 0
    # tiny shapes: one row, fewer rows than a block, one lane chunk of K
    for N, K in [(1, 128), (7, 128), (9, 256), (8, 1024), (13, 1152)]:
        yv, y_ref, b, _ = _gemm_case(fmt, group, 3, N, K, seed=N + K)
        assert ogemm.error_ratio(y_to_f64(yv), y_ref, b).max() <= 1.0, (N, K)
    # all-zero weights give exact zeros
    w = np.zeros((16, 256), dtype=np.float32)
    qz = oquant.quantize(w, fmt, group)
    wq, scales, zc = device_weights(qz, DEV)
    yz = uq.gemm(device_x(activations(5, 2, 256), DEV), wq, scales, zc, 16, group, fmt)
    assert torch.count_nonzero(yz.float()) == 0


def test_errors_on_device():
    xd = torch.zeros((1, 256), dtype=torch.bfloat16, device=DEV)
    wq = torch.zeros(256 * 128, dtype=torch.uint8, device=DEV)
    sc = torch.zeros(256 * 8, dtype=torch.int16, device=DEV)
    with pytest.raises(uq.UqError) as e:
        uq.gemm(xd, wq, sc, None, 256, 48, "INT4_SYM")
    assert e.value.status == 2
    with pytest.raises(uq.UqError) as e:
        uq.gemm(xd, wq, sc, sc, 256, 32, "INT4_SYM")
    assert e.value.status == 1


# ------------------------------------------------------------------------------------------
# full workload sizes: GPU quantizer on the whole weight, oracle on sampled rows

def _sample_rows(N, n=48, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(range(0, 8)) | set(range(N - 8, N)) | set(rng.integers(0, N, n).tolist())
    return np.array(sorted(rows))


def _full_case(fmt, group, N, K, M, seed, sigma, outliers):
    w = normal_weights(seed, N, K, sigma, outlier_p=0.001 if outliers else 0.0, outlier_mult=20.0)
    x = activations(seed, M, K)
    rows = _sample_rows(N, seed=seed)
    wd = torch.from_numpy(w).to(DEV)
    cb = nf4_codebook() if fmt == "NF4" else None
    if fmt == "K4":
        codes, d, dmin, sc, m = uq.quantize_k4(wd)
        scales = uq.pack_kmeta(d, dmin, sc, m)
        zc = None
        qz_rows = oquant.quantize_k4(w[rows])
        assert np.array_equal(codes[rows].cpu().numpy(), qz_rows.codes)
        assert np.array_equal(d[rows].cpu().numpy().view(np.uint16), qz_rows.d.view(np.uint16))
    else:
        cbd = torch.from_numpy(cb).to(DEV) if cb is not None else None
        codes, scales, zeros = uq.quantize(wd, group, fmt, codebook=cbd)
        qz_rows = oquant.quantize(w[rows], fmt, group, codebook=cb)
        assert np.array_equal(codes[rows].cpu().numpy(), qz_rows.codes)
        assert np.array_equal(scales[rows].cpu().numpy().view(np.uint16), qz_rows.scale.view(np.uint16))
        zc = uq.pack_zeros(zeros) if fmt == "INT4_ASYM" else (zeros if fmt == "INT2_ASYM" else cbd)
    del wd
    wq = uq.pack_layout(codes, group, fmt)
    y = uq.gemm(device_x(x, DEV), wq, scales, zc, N, group, fmt)
    y_ref, b = ogemm.reference(x, oquant.dequant(qz_rows))
    r = ogemm.error_ratio(y_to_f64(y)[:, rows], y_ref, b)
    assert r.max() <= 1.0, f"{fmt} {N}x{K} M={M}: max error ratio {r.max():.3g}"


@pytest.mark.parametrize("N,K", [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)])
def test_full_size_llama8b_linears_m1(N, K):
    _full_case("INT4_ASYM", 128, N, K, 1, seed=2000 + N + K, sigma=0.02, outliers=True)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_full_size_batched_sweep(N, K, M):
    _full_case("INT4_ASYM", 128, N, K, M, seed=3000 + M, sigma=0.02, outliers=False)


@pytest.mark.parametrize("fmt,group", [("INT8_SYM", 128), ("INT2_ASYM", 64), ("NF4", 64)])
@pytest.mark.parametrize("M", [1, 16])
def test_full_size_format_sweep(fmt, group, M):
    _full_case(fmt, group, 8192, 8192, M, seed=4000 + M, sigma=0.02, outliers=False)


@pytest.mark.parametrize("N,K", [(8192, 8192), (1024, 8192), (28672, 8192), (8192, 28672)])
@pytest.mark.parametrize("M", [1, 8, 32])
def test_full_size_k4_70b_linears(N, K, M):
    _full_case("K4", 256, N, K, M, seed=5000 + M, sigma=0.015, outliers=False)
