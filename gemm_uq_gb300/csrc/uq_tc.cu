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
    const int budget = 227 * 1024 - 1024 - TC_BAR_BYTES;
    int s = budget / (sb + TC_DQ_UNIT);
    if (s > 6) s = 6;
    if (s < 3) return -1;                           // codes are requested two units ahead
    int na = (TMEM_COLS - 2 * mpad) / (kc / 2);     // A buffers beside two Mpad-column accumulators
    if (na > 4) na = 4;
    if (na < 2) return -1;
    *stages = s;
    *nabuf = na;
    *smem = 1024 + (size_t)s * (sb + TC_DQ_UNIT) + TC_BAR_BYTES;
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

// Second pass when CTAs share 128-row blocks: y[m][n] = the sum of the contributing CTAs' partial
// sums in CTA order.  Launched right after the tensor-core kernel with programmatic stream
// serialization: its griddepcontrol.wait returns once that grid has finished and its stores are
// visible, so the kernel itself needs no fence or ticket.
__global__ void __launch_bounds__(256) tc_split_reduce(const TcArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int nblk = (a.N + TC_ROWS - 1) / TC_ROWS;
    const long long total = (long long)nblk * a.M * TC_ROWS;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int rb = (int)(e / ((long long)a.M * TC_ROWS));
        const int mr = (int)(e % ((long long)a.M * TC_ROWS));
        const int m = mr / TC_ROWS, r = mr % TC_ROWS;
        const int n = rb * TC_ROWS + r;
        if (n >= a.N) continue;
        const long long uf = (long long)rb * a.CH;
        const int cf = tworker_of(uf, a.U, a.P), cl = tworker_of(uf + a.CH - 1, a.U, a.P);
        if (cf == cl) continue;                                     // one CTA covered it and stored y
        float sum = 0.f;
        for (int c2 = cf; c2 <= cl; ++c2) {
            const int rb2 = (int)(trange_begin(c2, a.U, a.P) / a.CH);
            const int slot2 = 2 * c2 + (rb == rb2 ? 0 : 1);
            sum += a.partials[((long long)slot2 * a.Mpad + m) * TC_ROWS + r];
        }
        a.y[(long long)m * a.ldy + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
    }
}

// whether any 128-row block is shared by several CTAs (then the second pass runs)
static bool tc_any_split(const TcArgs& a) {
    const int nblk = (a.N + TC_ROWS - 1) / TC_ROWS;
    for (int rb = 0; rb < nblk; ++rb) {
        const long long uf = (long long)rb * a.CH, ul = uf + a.CH - 1;
        const long long cf = ((uf + 1) * a.P - 1) / a.U, cl = ((ul + 1) * a.P - 1) / a.U;
        if (cf != cl) return true;
    }
    return false;
}

static cudaError_t launch_tc_reduce(const TcArgs& a, int sms, cudaStream_t st) {
    const int nblk = (a.N + TC_ROWS - 1) / TC_ROWS;
    const long long total = (long long)nblk * a.M * TC_ROWS;
    long long blocks = (total + 255) / 256;
    if (blocks > 4LL * sms) blocks = 4LL * sms;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, tc_split_reduce, a);
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
    cudaError_t e;
    switch (fmt) {
        case UQ_INT4_SYM: e = launch_tc_fmt<UQ_INT4_SYM>(mx, a, smem, grid, st); break;
        case UQ_INT4_ASYM: e = launch_tc_fmt<UQ_INT4_ASYM>(mx, a, smem, grid, st); break;
        case UQ_INT8_SYM: e = launch_tc_fmt<UQ_INT8_SYM>(mx, a, smem, grid, st); break;
        case UQ_K4: e = launch_tc_fmt<UQ_K4>(mx, a, smem, grid, st); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess || !tc_any_split(a)) return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return launch_tc_reduce(a, sms > 0 ? sms : 1, st);
}

}  // namespace uq
