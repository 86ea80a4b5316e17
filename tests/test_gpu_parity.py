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
from tests.uq_helpers import mma_gemm_launches, KT, device_weights, device_x, h16, y_to_f64  # noqa: E402

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
    # 14336 x 4096 at M = 1: whole row blocks per CTA, one launch; 4096 x 14336 too (4 tiles a warp
    # against 3 under the split, one launch fewer); 1024 x 14336: the stream-K split (a partial-sum
    # slot per tile) and its second pass; M >= 16: the tensor cores per 64 rows; 9..15 rows and K4:
    # the mma.sync GEMM (a split k range adds its second pass, K4 its x column-sum pre-kernel); NF4
    # with a K that is not a multiple of the code tile keeps M = 20 on the GEMV: three 8-row blocks
    assert uq.gemm_kernel_count(1, 14336, 4096, 128, "INT4_ASYM") == 1
    assert uq.gemm_noalloc_scratch(1, 14336, 4096, 128, "INT4_ASYM") == (0, 0)
    assert uq.gemm_kernel_count(1, 4096, 14336, 128, "INT4_ASYM") == 1
    assert uq.gemm_noalloc_scratch(1, 4096, 14336, 128, "INT4_ASYM") == (0, 0)
    assert uq.gemm_kernel_count(1, 1024, 14336, 128, "INT4_ASYM") == 2
    assert uq.gemm_noalloc_scratch(1, 1024, 14336, 128, "INT4_ASYM") == (0, 64 * 14 * 16 * 4)
    # INT8 8192 x 8192 at M = 1 (512-k tiles): whole row blocks would give a CTA 64 tiles, more than
    # it holds partial sums for, so the stream-K split and its second pass
    assert uq.gemm_kernel_count(1, 8192, 8192, 128, "INT8_SYM") == 2
    assert uq.gemm_noalloc_scratch(1, 8192, 8192, 128, "INT8_SYM") == (0, 512 * 16 * 16 * 4)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert uq.gemm_kernel_count(64, 14336, 4096, 128, "INT4_ASYM") == 1
    assert uq.gemm_kernel_count(128, 14336, 4096, 128, "INT4_ASYM") == 2
    assert uq.gemm_kernel_count(9, 14336, 4096, 128, "INT4_ASYM") == mma_gemm_launches("INT4_ASYM", 14336, 4096, sms)
    assert uq.gemm_kernel_count(32, 8192, 8192, 256, "K4") == mma_gemm_launches("K4", 8192, 8192, sms)
    assert uq.gemm_kernel_count(20, 4096, 4096, 64, "NF4") == 1
    assert uq.gemm_kernel_count(20, 4096, 4096 + 64, 64, "NF4") == 3      # K not a multiple of the tile


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
# full workload sizes: every output element of every M against the oracle.  The weight is quantized
# on the GPU (the library's quantizer) and by the oracle in row blocks (to bound host memory); the
# two must agree bit for bit on every row, and every row of y is checked against the oracle's
# float64 dequantize-then-matmul of its own quantization.

ORACLE_ROWS = 2048


def _oracle_rows(w, fmt, group, cb, r0, r1):
    if fmt == "K4":
        return oquant.quantize_k4(w[r0:r1])
    return oquant.quantize(w[r0:r1], fmt, group, codebook=cb)


def _full_shape(fmt, group, N, K, Ms, seed, sigma, outliers):
    w = normal_weights(seed, N, K, sigma, outlier_p=0.001 if outliers else 0.0, outlier_mult=20.0)
    xs = {M: activations(seed + 7919 * M, M, K) for M in Ms}
    wd = torch.from_numpy(w).to(DEV)
    cb = nf4_codebook() if fmt == "NF4" else None
    if fmt == "K4":
        codes, d, dmin, sc, m = uq.quantize_k4(wd)
        scales = uq.pack_kmeta(d, dmin, sc, m)
        zc = None
        gpu_meta = {"d": d.cpu().numpy().view(np.uint16), "dmin": dmin.cpu().numpy().view(np.uint16),
                    "sc": sc.cpu().numpy(), "m": m.cpu().numpy()}
        del d, dmin, sc, m
    else:
        cbd = torch.from_numpy(cb).to(DEV) if cb is not None else None
        codes, scales, zeros = uq.quantize(wd, group, fmt, codebook=cbd)
        gpu_meta = {"scale": scales.cpu().numpy().view(np.uint16)}
        if fmt == "INT4_ASYM":
            gpu_meta["zero"] = zeros.cpu().numpy()
        if fmt == "INT2_ASYM":
            gpu_meta["zero"] = zeros.cpu().numpy().view(np.uint16)
        zc = uq.pack_zeros(zeros) if fmt == "INT4_ASYM" else (zeros if fmt == "INT2_ASYM" else cbd)
    del wd
    gpu_codes = codes.cpu().numpy()
    wq = uq.pack_layout(codes, group, fmt)
    del codes
    ys = {M: y_to_f64(uq.gemm(device_x(xs[M], DEV), wq, scales, zc, N, group, fmt)) for M in Ms}
    worst = {M: 0.0 for M in Ms}
    for r0 in range(0, N, ORACLE_ROWS):
        r1 = min(N, r0 + ORACLE_ROWS)
        qz = _oracle_rows(w, fmt, group, cb, r0, r1)
        assert np.array_equal(gpu_codes[r0:r1], qz.codes), f"GPU codes differ in rows {r0}..{r1}"
        if fmt == "K4":
            assert np.array_equal(gpu_meta["d"][r0:r1], qz.d.view(np.uint16))
            assert np.array_equal(gpu_meta["dmin"][r0:r1], qz.dmin.view(np.uint16))
            assert np.array_equal(gpu_meta["sc"][r0:r1], qz.sc)
            assert np.array_equal(gpu_meta["m"][r0:r1], qz.m)
        else:
            assert np.array_equal(gpu_meta["scale"][r0:r1], qz.scale.view(np.uint16))
            if fmt == "INT4_ASYM":
                assert np.array_equal(gpu_meta["zero"][r0:r1], qz.zero)
            if fmt == "INT2_ASYM":
                assert np.array_equal(gpu_meta["zero"][r0:r1], qz.zero.view(np.uint16))
        w_hat = oquant.dequant(qz)
        for M in Ms:
            y_ref, b = ogemm.reference(xs[M], w_hat)
            r = ogemm.error_ratio(ys[M][:, r0:r1], y_ref, b)
            worst[M] = max(worst[M], float(r.max()))
    for M in Ms:
        assert worst[M] <= 1.0, f"{fmt} {N}x{K} M={M}: max error ratio {worst[M]:.3g}"


@pytest.mark.parametrize("N,K", [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)])
def test_full_size_llama8b_linears_m1(N, K):
    _full_shape("INT4_ASYM", 128, N, K, [1], seed=2000 + N + K, sigma=0.02, outliers=True)


@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_full_size_batched_sweep(N, K):
    _full_shape("INT4_ASYM", 128, N, K, [1, 2, 4, 8, 16, 32, 64], seed=3000 + N // 1024, sigma=0.02,
                outliers=False)


@pytest.mark.parametrize("fmt,group", [("INT8_SYM", 128), ("INT2_ASYM", 64), ("NF4", 64)])
def test_full_size_format_sweep(fmt, group):
    _full_shape(fmt, group, 8192, 8192, [1, 16], seed=4000 + group, sigma=0.02, outliers=False)


@pytest.mark.parametrize("N,K", [(8192, 8192), (1024, 8192), (28672, 8192), (8192, 28672)])
def test_full_size_k4_70b_linears(N, K):
    _full_shape("K4", 256, N, K, [1, 8, 32], seed=5000 + N // 1024 + K // 1024, sigma=0.015, outliers=False)


# ------------------------------------------------------------------------------------------
# fp16 subnormal d and dmin in K4 records: decoded exactly by the dequant export and the GEMM paths

def _subnormal_k4(N, K, seed):
    """Hand-set K4 weights whose every super-block has an fp16 subnormal d and dmin (bit patterns
    1..1023), full-range 6-bit sc and m, and random 4-bit codes: the decode must be exact there."""
    rng = np.random.default_rng(seed)
    S = K // 256
    d = rng.integers(1, 1024, (N, S)).astype(np.uint16).view(np.float16)
    dmin = rng.integers(1, 1024, (N, S)).astype(np.uint16).view(np.float16)
    d[0, 0] = np.uint16(1).view(np.float16)            # the smallest subnormal
    dmin[0, 0] = np.uint16(0x03FF).view(np.float16)    # the largest subnormal
    sc = rng.integers(0, 64, (N, S, 8)).astype(np.uint8)
    m = rng.integers(0, 64, (N, S, 8)).astype(np.uint8)
    sc[0, 0, :2] = (63, 0)
    m[0, 0, :2] = (0, 63)
    codes = rng.integers(0, 16, (N, K)).astype(np.int8)
    return oquant.Quantized("K4", 256, codes, d=d, dmin=dmin, sc=sc, m=m)


def test_k4_subnormal_d_dmin_dequant_bit_exact():
    qz = _subnormal_k4(48, 1024, 61)
    assert np.all(np.abs(qz.d.astype(np.float64)) < 2.0 ** -14)
    assert np.all(np.abs(qz.dmin.astype(np.float64)) < 2.0 ** -14)
    wq, scales, zc = device_weights(qz, DEV)
    got = uq.dequant(wq, scales, zc, 48, 1024, 256, "K4").cpu().numpy()
    want = oquant.dequant(qz)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("M", [1, 8, 32])
def test_k4_subnormal_d_dmin_gemm(M):
    N, K = 300, 2048
    qz = _subnormal_k4(N, K, 62)
    x = activations(63, M, K)
    wq, scales, zc = device_weights(qz, DEV)
    y = uq.gemm(device_x(x, DEV), wq, scales, zc, N, 256, "K4")
    y_ref, b = ogemm.quantized_gemm(x, qz)
    r = ogemm.error_ratio(y_to_f64(y), y_ref, b)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3g}"
