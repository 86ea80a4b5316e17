// uq_w4a8.cu -- W4A8 / W8A8: dynamic per-row int8 activations and integer dot products (sm_103a).
//
// "Ultra LLM Engine", section "Quantized Model": the activations are dynamically quantized for the
// GEMV/GEMM paths.  Per row m of x: s_x = absmax / 127 (fp32), xq = clamp(RNE(x / s_x), -127, 127)
// (fp32 quotient); then y[m][n] = s_x * sum_g s[n][g] * I, I = sum_{k in g} xq * (q - z), an exact
// integer formed on the integer tensor instructions (mma.m16n8k32, u8 x s8 -> s32).
//
// quant_x_kernel (a cluster of 8 CTAs per row): absmax, s_x, the codes, written with each 4-k group's bytes in the
// order the weight words hold their codes (4-bit: k, k+2, k+1, k+3 -- the low nibbles of a fragment-
// order word; 8-bit: k .. k+3) and the 4-k groups placed in the integer mma's B fragment order, and per
// group the sum of its codes, for the zero-point term.
// The integer GEMV (gemv_mma_kernel's A8 mode, csrc/uq_gemv.cuh): the decode GEMV's copy-warp ring and
// work split (whole row blocks per CTA, or the stream-K split and its second pass), with an integer
// tensor-core inner loop: per pair of 16-k blocks a lane takes its two code words, masks the two rows'
// codes into bytes (w & 0x0F0F0F0F, (w >> 4) & 0x0F0F0F0F for 4-bit; INT8 words are already bytes) --
// the A fragment of mma.m16n8k32 (u8 x s8 -> s32) -- and one instruction forms the exact integer sums
// of 16 weight rows x 8 rows of x over 32 k.  Per group: acc += s * (D - zc * SX), zc the stored
// code's offset (8 for INT4_SYM, z for INT4_ASYM, 128 for INT8_SYM); each tile's sums times s_x.
#include "uq_gemv.cuh"

namespace uq {

namespace {


// One cluster of QX_CTAS CTAs (QX_THREADS threads each) per row of x; CTA r of the cluster takes a
// contiguous share of the row's 8-k segments (a multiple of 16 segments, so no scaling group spans
// two CTAs).  Each thread takes 8 consecutive k at a time (one 16-byte load of x): first the share's
// absmax, which the cluster combines through distributed shared memory into the row's absmax, then
// per 8 k the codes (two 4-k groups, each written as one word at its place in the B fragment order)
// and their sum, which a shuffle tree adds up over the gs / 8 lanes of a scaling group (consecutive
// lanes of one warp).  Integer sums: any order gives the same result.
constexpr int QX_THREADS = 256;
constexpr int QX_CTAS = 8;
__global__ void __launch_bounds__(QX_THREADS) quant_x_kernel(const uint16_t* __restrict__ x, int8_t* __restrict__ xq,
                                                             float* __restrict__ sx, int* __restrict__ sxl, int M,
                                                             int K, int Kp, int gs, int perm) {
    __shared__ float red[QX_THREADS / 32];
    __shared__ float share_max;
    // the GEMV that reads these codes may start streaming its (constant) weights meanwhile; its
    // griddepcontrol.wait returns once this grid has finished
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int m = blockIdx.y;
    const int r = blockIdx.x;                                       // rank in the row's cluster
    const int nseg = Kp / 8;
    const int per = ((nseg + QX_CTAS - 1) / QX_CTAS + 15) / 16 * 16;
    const int seg0 = r * per, seg1 = (seg0 + per) < nseg ? (seg0 + per) : nseg;
    const uint16_t* xr = x + (long long)m * K;
    // K is a multiple of the group (>= 32), so whole 8-k segments: one 16-byte load each (x rows are
    // 16-byte aligned: the row start and K * 2 are multiples of 16)
    float mx = 0.f;
    for (int sg = seg0 + threadIdx.x; sg < seg1 && sg * 8 < K; sg += QX_THREADS) {
        const uint4 v = *reinterpret_cast<const uint4*>(xr + sg * 8);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.f;
        for (int w = 0; w < QX_THREADS / 32; ++w) b = fmaxf(b, red[w]);
        share_max = b;
    }
    // every CTA's share_max is written before any CTA reads them
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    float amax = 0.f;
    for (int q = 0; q < QX_CTAS; ++q) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(&share_max)), "r"(q));
        float v;
        asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
        amax = fmaxf(amax, v);
    }
    const float s = __fdiv_rn(amax, 127.0f);
    if (threadIdx.x == 0 && r == 0) sx[m] = s;
    // codes in the weight words' byte order, placed in the B fragment order of the integer mma:
    // per 32 k and lane column c, the 4 codes of k = 32t + 4c .. then those of k = 32t + 16 + 4c ..
    // (8 contiguous bytes, one load per instruction)
    int8_t* qr = xq + (long long)m * Kp;
    const int G = (Kp + gs - 1) / gs;
    const int lpg = gs / 8;                                         // lanes per scaling group
    for (int base = seg0; base < seg1; base += QX_THREADS) {       // the same trip count on every lane
        const int sg = base + threadIdx.x;
        const int k8 = sg * 8;
        int tot = 0;
        if (sg < seg1) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (k8 < K) v = *reinterpret_cast<const uint4*>(xr + k8);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {                           // the two 4-k groups
                int q[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t wd = w[2 * h + (j >> 1)];
                    const float xv = __uint_as_float((j & 1) ? (wd & 0xFFFF0000u) : (wd << 16));
                    float c = 0.f;
                    if (k8 + 4 * h + j < K && s > 0.f) c = rintf(__fdiv_rn(xv, s));
                    c = fminf(fmaxf(c, -127.f), 127.f);
                    q[j] = (int)c;
                    tot += q[j];
                }
                const uint32_t packed = perm ? ((uint32_t)(q[0] & 255) | ((uint32_t)(q[2] & 255) << 8) |
                                                ((uint32_t)(q[1] & 255) << 16) | ((uint32_t)(q[3] & 255) << 24))
                                             : ((uint32_t)(q[0] & 255) | ((uint32_t)(q[1] & 255) << 8) |
                                                ((uint32_t)(q[2] & 255) << 16) | ((uint32_t)(q[3] & 255) << 24));
                const int k4 = k8 + 4 * h;
                const int blk = k4 >> 4, cc = (k4 >> 2) & 3;
                *reinterpret_cast<uint32_t*>(qr + (blk >> 1) * 32 + cc * 8 + (blk & 1) * 4) = packed;
            }
        }
        // the group's sum over its lpg lanes (seg0 and the step are multiples of lpg, so a group's
        // segments sit on consecutive lanes starting at a multiple of lpg)
        for (int o = 1; o < lpg; o <<= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if (sg < seg1 && (sg % lpg) == 0) sxl[(long long)m * G + k8 / gs] = tot;
    }
    // no CTA leaves while a peer may still read its share_max
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace

cudaError_t launch_quant_x(const uint16_t* x, int8_t* xq, float* sx, int* sxl, int M, int K, int Kp, int gs, int perm,
                           cudaStream_t st) {
    const int G = (Kp + gs - 1) / gs;
    for (int m0 = 0; m0 < M; m0 += 65535) {                        // rows per launch: the grid's y extent
        const int mb = (M - m0) < 65535 ? (M - m0) : 65535;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(QX_CTAS, (unsigned)mb);
        cfg.blockDim = dim3(QX_THREADS);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = QX_CTAS;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, quant_x_kernel, x + (long long)m0 * K, xq + (long long)m0 * Kp, sx + m0,
                                           sxl + (long long)m0 * G, mb, K, Kp, gs, perm);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

// The integer GEMV is gemv_mma_kernel's A8 mode (csrc/uq_gemv.cuh): the copy-warp ring of tile
// pairs, the CTA's window of x codes in shared memory, the integer group step.
cudaError_t launch_gemv_a8(int fmt, const GemvArgs& a, const int8_t* xq, const float* sxs, const int* sxl, int Kp,
                           int grid, cudaStream_t st) {
    GemvArgs b = a;
    b.xq = xq;
    b.sxq = sxs;
    b.sxl = sxl;
    b.Kpq = Kp;
    cudaError_t e = cudaErrorInvalidValue;
    const int gb = a.group / 16;
    switch (fmt) {
        case UQ_INT4_SYM:
            e = gb == 2 ? gemv_detail::launch_mma_x<UQ_INT4_SYM, 2, false, true>(b, grid, st)
              : gb == 4 ? gemv_detail::launch_mma_x<UQ_INT4_SYM, 4, false, true>(b, grid, st)
              : gb == 8 ? gemv_detail::launch_mma_x<UQ_INT4_SYM, 8, false, true>(b, grid, st) : cudaErrorInvalidValue;
            break;
        case UQ_INT4_ASYM:
            e = gb == 2 ? gemv_detail::launch_mma_x<UQ_INT4_ASYM, 2, false, true>(b, grid, st)
              : gb == 4 ? gemv_detail::launch_mma_x<UQ_INT4_ASYM, 4, false, true>(b, grid, st)
              : gb == 8 ? gemv_detail::launch_mma_x<UQ_INT4_ASYM, 8, false, true>(b, grid, st) : cudaErrorInvalidValue;
            break;
        case UQ_INT8_SYM:
            e = gb == 2 ? gemv_detail::launch_mma_x<UQ_INT8_SYM, 2, false, true>(b, grid, st)
              : gb == 4 ? gemv_detail::launch_mma_x<UQ_INT8_SYM, 4, false, true>(b, grid, st)
              : gb == 8 ? gemv_detail::launch_mma_x<UQ_INT8_SYM, 8, false, true>(b, grid, st) : cudaErrorInvalidValue;
            break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess || a.cta_rows) return e;
    return launch_gemv_second_pass(a, grid, st);
}

}  // namespace uq
