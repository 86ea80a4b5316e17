// uq_tc.cu -- host side of the tensor-core path (uq_tc.cuh): the x pre-kernel, the shared-memory
// plan, the x tensor map and the per-format dispatch.
//
// "Ultra LLM Engine", section "Fused Kernels": the dequantized-weight GEMM of batched decode.
#include "uq_tc.cuh"

namespace uq {

extern template cudaError_t launch_tc_fmt<UQ_INT4_SYM>(const CUtensorMap&, const TcArgs&, size_t, int, cudaStream_t);
extern template cudaError_t launch_tc_fmt<UQ_INT4_ASYM>(const CUtensorMap&, const TcArgs&, size_t, int, cudaStream_t);
extern template cudaError_t launch_tc_fmt<UQ_INT8_SYM>(const CUtensorMap&, const TcArgs&, size_t, int, cudaStream_t);
extern template cudaError_t launch_tc_fmt<UQ_K4>(const CUtensorMap&, const TcArgs&, size_t, int, cudaStream_t);

// x row m (bf16) -> fp16 scaled by 2^-e_m, e_m chosen from the row's largest magnitude so that it
// lands in [2^14, 2^15) (a power-of-two scale is exact; the epilogue multiplies by 2^e_m).
// One CTA per row; xs[m] = 2^e_m, and xs[M .. mpad) = 0 for the padding columns.
__global__ void __launch_bounds__(256) tc_prep_x_kernel(const uint16_t* __restrict__ x, int ldx, int K, int M, int mpad,
                                                         uint16_t* __restrict__ xh, float* __restrict__ xs) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int m = blockIdx.x;
    const uint16_t* row = x + (long long)m * ldx;
    __shared__ unsigned int red[8];
    unsigned int mx = 0;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const unsigned int v = row[k] & 0x7FFFu;                   // |x| as bits: monotonic for finite values
        mx = v > mx ? v : mx;
    }
    for (int o = 16; o; o >>= 1) {
        const unsigned int t = __shfl_xor_sync(0xffffffffu, mx, o);
        mx = t > mx ? t : mx;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0;
    for (int i = 0; i < 8; ++i) mx = red[i] > mx ? red[i] : mx;
    int e = 0;
    const int E = (int)(mx >> 7);                                   // bf16 biased exponent of the max
    if (mx != 0 && E < 255) e = (E - 127) - 14;
    if (e < -100) e = -100;
    const float down = exp2f((float)(-e)), up = exp2f((float)e);    // exact powers of two
    for (int k = threadIdx.x; k < K; k += blockDim.x)
        xh[(long long)m * K + k] = __half_as_ushort(__float2half_rn(__uint_as_float((uint32_t)row[k] << 16) * down));
    if (threadIdx.x == 0) xs[m] = up;
    if (m == 0)
        for (int j = M + threadIdx.x; j < mpad; j += blockDim.x) xs[j] = 0.f;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}
}  // namespace

bool tc_supported(int fmt, int N, int K) {
    if (fmt != UQ_INT4_SYM && fmt != UQ_INT4_ASYM && fmt != UQ_INT8_SYM && fmt != UQ_K4) return false;
    if (N < 1 || K % fmt_kt(fmt)) return false;
    return encode_fn() != nullptr;
}

int tc_plan(int fmt, int mpad, int* stages, int* nabuf, size_t* smem) {
    const int kc = (fmt == UQ_INT8_SYM) ? 128 : 256;
    const int sb = TcSmem::stage_bytes(kc, mpad);
    const int budget = 227 * 1024 - 1024 - TC_BAR_BYTES - TC_DQ_RING;
    int s = budget / sb;
    if (s > 6) s = 6;
    if (s < 2) return -1;
    int na = (TMEM_COLS - 2 * mpad) / (kc / 2);     // A buffers beside two Mpad-column accumulators
    if (na > 4) na = 4;
    if (na < 2) return -1;
    *stages = s;
    *nabuf = na;
    *smem = 1024 + (size_t)s * sb + TC_BAR_BYTES + TC_DQ_RING;
    return 0;
}

cudaError_t launch_tc_prep(const uint16_t* x, int ldx, int K, int M, int mpad, uint16_t* xh, float* xs,
                           cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(M);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = launch_overlap() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, tc_prep_x_kernel, x, ldx, K, M, mpad, xh, xs);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_tc(int fmt, const uint16_t* xh, const TcArgs& a, size_t smem, int grid, cudaStream_t st) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap mx;
    {
        cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
        cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)a.Mpad};
        cuuint32_t es[2] = {1, 1};
        if (enc(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(xh), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    switch (fmt) {
        case UQ_INT4_SYM: return launch_tc_fmt<UQ_INT4_SYM>(mx, a, smem, grid, st);
        case UQ_INT4_ASYM: return launch_tc_fmt<UQ_INT4_ASYM>(mx, a, smem, grid, st);
        case UQ_INT8_SYM: return launch_tc_fmt<UQ_INT8_SYM>(mx, a, smem, grid, st);
        case UQ_K4: return launch_tc_fmt<UQ_K4>(mx, a, smem, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace uq
