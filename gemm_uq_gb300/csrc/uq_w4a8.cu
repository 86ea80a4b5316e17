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
// gemv_a8_kernel: the decode GEMV's tiles, copy rings and work split (whole row blocks per CTA, or the
// stream-K split and its second pass), with an integer tensor-core inner loop: per pair of 16-k blocks
// a lane takes its two code words, masks the two rows' codes into bytes (w & 0x0F0F0F0F,
// (w >> 4) & 0x0F0F0F0F for 4-bit; INT8 words are already bytes) -- the A fragment of
// mma.m16n8k32 (u8 x s8 -> s32) -- and one instruction forms the exact integer sums of 16 weight
// rows x 8 rows of x over 32 k.  Per group: acc += s * (D - zc * SX), zc the stored code's offset
// (8 for INT4_SYM, z for INT4_ASYM, 128 for INT8_SYM).
#include "uq_gemv.cuh"

namespace uq {

namespace {

// D += A * B for one 16 x 8 x 32 block: A unsigned 8-bit (the stored codes), B signed 8-bit (x codes),
// exact 32-bit integer accumulation
__device__ __forceinline__ void mma_u8s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

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

// Shared memory of the A8 GEMV: rings [warps][stages][stage] | ring mbarriers | partial sums
template <int FMT>
__host__ __device__ inline GemvSmem gemv_a8_smem_plan() {
    using F = GemvFmt<FMT>;
    constexpr int W = 4, S = 2;
    GemvSmem p;
    p.bars = (size_t)W * S * MetaGeom<FMT>::STAGE_BYTES;
    p.lut = p.bars + (size_t)W * S * 8;
    p.sx = p.lut;
    p.ps = (p.lut + 15) / 16 * 16;
    p.x = p.ps + (size_t)W * A8_TPW * RB * 8 * 4;
    p.total = p.x;
    return p;
}

// GB = 16-k blocks per scaling group
template <int FMT, int GB>
__global__ void __launch_bounds__(128, A8_CTAS_PER_SM) gemv_a8_kernel(const GemvArgs a, const int8_t* __restrict__ xq,
                                                                       const float* __restrict__ sxs,
                                                                       const int* __restrict__ sxl, int Kp) {
    using F = GemvFmt<FMT>;
    constexpr int KT = F::KT, S = 2, W = 4;
    constexpr int GS = GB * 16, GPT = KT / GS;
    constexpr int BPCH = F::BPC;                                    // 16-k blocks per 512-byte chunk
    extern __shared__ __align__(128) uint8_t smem[];
    const int M = a.M;
    const GemvSmem plan = gemv_a8_smem_plan<FMT>();
    float* cpart = reinterpret_cast<float*>(smem + plan.ps);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const Layout L(a.N, a.K, FMT);
    uint8_t* ring = smem + (size_t)warp * S * MetaGeom<FMT>::STAGE_BYTES;

    // work split as the mma GEMV's (k-major tiles; whole row blocks per CTA, or stream-K)
    const bool cta_rows = a.cta_rows != 0;
    const int rb0 = cta_rows ? (int)((long long)blockIdx.x * a.NB / gridDim.x) : 0;
    const int R = cta_rows ? (int)((long long)(blockIdx.x + 1) * a.NB / gridDim.x) - rb0 : a.NB;
    const unsigned Tc = (unsigned)(R * L.KB);
    const int w = cta_rows ? warp : (int)(blockIdx.x + gridDim.x * warp);
    const bool has_work = cta_rows ? true : w < a.P;
    const long long t0 = cta_rows ? (long long)(warp * Tc / W) : (has_work ? range_begin(w, a.T, a.P) : 0);
    const long long t1 = cta_rows ? (long long)((warp + 1) * Tc / W) : (has_work ? range_begin(w + 1, a.T, a.P) : 0);
    int ntl = (int)(t1 - t0);
    if (cta_rows && ntl > A8_TPW) {
        if (lane == 0) atomicOr(a.fault, FAULT_GEMV_SPLIT);
        ntl = 0;
    }
    auto kb_of = [&](long long i) { return (int)(i / R); };
    auto nb_of = [&](long long i) { return rb0 + (int)(i % R); };
    MetaConst mc;
    mc.G = a.K / a.group;
    mc.GT = KT / a.group;
    mc.ZB = (mc.G + 1) >> 1;
    mc.S4 = a.K / 256;
    mc.aligned = (a.K % (8 * a.group)) == 0 && (mc.GT % 8) == 0;
    const int G_all = a.K / GS;
    const int Gq = (Kp + GS - 1) / GS;                              // groups of the code-sum table
    const GemvSrc src{a.wq, a.scales, a.zc};

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int issued = 0;
    // k-major tile coordinates advanced incrementally (no 64-bit division per tile)
    int ikb = ntl > 0 ? kb_of(t0) : 0, irb = ntl > 0 ? (int)(t0 % R) : 0;   // the next tile to request
    auto issue_next = [&]() {
        issue_tile<FMT, GPT>(a, src, L, mc, rb0 + irb, ikb, ring + (issued % S) * MetaGeom<FMT>::STAGE_BYTES, lane);
        if (++irb == R) { irb = 0; ++ikb; }
        ++issued;
    };
    if (a.overlap && has_work && ntl > 0) issue_next();           // weights are constant: before the wait
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (has_work && issued == 0 && ntl > 0) issue_next();
    if (!has_work) return;

    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};   // rows g + 8 jr, columns 2c + e
    float sxm[2];                                 // the scales of x of columns 2c, 2c + 1
#pragma unroll
    for (int e = 0; e < 2; ++e) sxm[e] = 2 * c + e < M ? __ldg(sxs + 2 * c + e) : 0.f;

    int ckb = ntl > 0 ? kb_of(t0) : 0, crb = ntl > 0 ? (int)(t0 % R) : 0;   // the tile being consumed
    for (int li = 0; li < ntl; ++li) {
        const long long i = t0 + li;
        const int kb = ckb, nb = rb0 + crb;
        if (++crb == R) { crb = 0; ++ckb; }
        const int n0 = nb * RB;
        const int gi0 = kb * GPT;
        const int ng = (G_all - gi0) < GPT ? (G_all - gi0) : GPT;
        while (issued < ntl && issued < li + S) issue_next();
        const int s = li % S;
        uint8_t* st = ring + s * MetaGeom<FMT>::STAGE_BYTES;
        if (issued > li + 1) cp_async_wait_group<1>();
        else cp_async_wait_group<0>();
        __syncwarp();
        RowPtrs<FMT> rp[2];
        rp[0] = row_ptrs<FMT>(st, mc, g, n0 + g, kb);
        rp[1] = row_ptrs<FMT>(st, mc, g + 8, n0 + g + 8, kb);
        // lane (g, c): rows g, g + 8 of D; columns (rows of x) 2c, 2c + 1
        const int m0c = 2 * c < M ? 2 * c : M - 1, m1c = 2 * c + 1 < M ? 2 * c + 1 : M - 1;
        const uint8_t* xg = reinterpret_cast<const uint8_t*>(xq) + (long long)(g < M ? g : M - 1) * Kp + 8 * c;
        auto group_step = [&](const int gg) {
            // the group's exact integer sum of (stored code) x (x code) per row and column: GB / 2
            // instructions of m16n8k32 (u8 x s8 -> s32), each over two 16-k blocks
            int d[4] = {0, 0, 0, 0};
#pragma unroll
            for (int t = 0; t < GB / 2; ++t) {
                const int blk = gg * GB + 2 * t;                    // even block of the pair, within the tile
                uint32_t a0, a1, a2, a3;
                if constexpr (FMT == UQ_INT8_SYM) {
                    // one chunk = the pair: row g, row g + 8 of the even block, then of the odd one
                    const uint4 v = *reinterpret_cast<const uint4*>(st + (blk / BPCH) * CHUNK + lane * 16);
                    a0 = v.x; a1 = v.y; a2 = v.z; a3 = v.w;
                } else {
                    const uint2 v = *reinterpret_cast<const uint2*>(st + (blk / BPCH) * CHUNK + lane * 16 + (blk % BPCH) * 4);
                    a0 = v.x & 0x0F0F0F0Fu;                         // row g:     k, k+2, k+1, k+3
                    a1 = (v.x >> 4) & 0x0F0F0F0Fu;                  // row g + 8: the same order
                    a2 = v.y & 0x0F0F0F0Fu;
                    a3 = (v.y >> 4) & 0x0F0F0F0Fu;
                }
                // x codes of the pair for column g, stored in this fragment's order
                const uint2 bv = *reinterpret_cast<const uint2*>(xg + (long long)(kb * KT + blk * 16));
                mma_u8s8(d, a0, a1, a2, a3, bv.x, bv.y);
            }
            // fold the group: acc += s * (D - zc * SX), SX the sum of the group's x codes of the column
            const int gi = gi0 + gg;
            const int sx0 = __ldg(sxl + (long long)m0c * Gq + gi), sx1 = __ldg(sxl + (long long)m1c * Gq + gi);
#pragma unroll
            for (int jr = 0; jr < 2; ++jr) {
                float sc, zcf;
                row_meta<FMT>(rp[jr], gg, sc, zcf);               // 4-bit: zcf = 128 + the stored code offset
                const int zc = (FMT == UQ_INT8_SYM) ? 128 : (int)zcf - 128;   // INT8 codes are stored + 128
                acc[jr][0] = fmaf(sc, (float)(d[2 * jr] - zc * sx0), acc[jr][0]);
                acc[jr][1] = fmaf(sc, (float)(d[2 * jr + 1] - zc * sx1), acc[jr][1]);
            }
        };
        if (ng == GPT) {
            // whole tiles: several groups' loads (codes, x codes, their sums) in flight together
#pragma unroll 4
            for (int gg = 0; gg < GPT; ++gg) group_step(gg);
        } else {
#pragma unroll 1
            for (int gg = 0; gg < ng; ++gg) group_step(gg);
        }
        __syncwarp();
        // the tile's partial sums (rows g + 8 jr, columns 2c + e), stored like the mma GEMV's
#pragma unroll
        for (int jr = 0; jr < 2; ++jr)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int m = 2 * c + e;
                const float v = acc[jr][e] * sxm[e];
                acc[jr][e] = 0.f;
                if (m >= M) continue;
                if (cta_rows) cpart[(i * RB + g + 8 * jr) * 8 + m] = v;   // slot = the tile's index in the CTA's range
                else a.partials[(i * RB + g + 8 * jr) * M + m] = v;
            }
    }
    cp_async_wait_group<0>();
    if (!cta_rows) return;
    __syncthreads();
    for (int e = threadIdx.x; e < R * RB * M; e += blockDim.x) {
        const int rbi = e / (RB * M), rm = e % (RB * M), r = rm / M, m = rm % M;
        const int n = (rb0 + rbi) * RB + r;
        if (n >= a.N) continue;
        float sum = 0.f;
        for (int kbb = 0; kbb < L.KB; ++kbb) sum += cpart[((kbb * R + rbi) * RB + r) * 8 + m];
        store_out(a, m, n, sum);
    }
}

namespace {
template <int FMT, int GB>
cudaError_t launch_a8_t(const GemvArgs& a, const int8_t* xq, const float* sxs, const int* sxl, int Kp, int grid,
                        cudaStream_t st) {
    static bool configured[64] = {};
    const size_t smem = gemv_a8_smem_plan<FMT>().total;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gemv_a8_kernel<FMT, GB>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    GemvArgs a2 = a;
    a2.overlap = launch_overlap() ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a2.overlap ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, gemv_a8_kernel<FMT, GB>, a2, xq, sxs, sxl, Kp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}
template <int FMT>
cudaError_t launch_a8_f(const GemvArgs& a, const int8_t* xq, const float* sxs, const int* sxl, int Kp, int grid,
                        cudaStream_t st) {
    switch (a.group) {
        case 32: return launch_a8_t<FMT, 2>(a, xq, sxs, sxl, Kp, grid, st);
        case 64: return launch_a8_t<FMT, 4>(a, xq, sxs, sxl, Kp, grid, st);
        case 128: return launch_a8_t<FMT, 8>(a, xq, sxs, sxl, Kp, grid, st);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

size_t a8_smem_bytes(int fmt) {
    switch (fmt) {
        case UQ_INT4_SYM: return gemv_a8_smem_plan<UQ_INT4_SYM>().total;
        case UQ_INT4_ASYM: return gemv_a8_smem_plan<UQ_INT4_ASYM>().total;
        default: return gemv_a8_smem_plan<UQ_INT8_SYM>().total;
    }
}

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

cudaError_t launch_gemv_a8(int fmt, const GemvArgs& a, const int8_t* xq, const float* sxs, const int* sxl, int Kp,
                           int grid, cudaStream_t st) {
    cudaError_t e;
    switch (fmt) {
        case UQ_INT4_SYM: e = launch_a8_f<UQ_INT4_SYM>(a, xq, sxs, sxl, Kp, grid, st); break;
        case UQ_INT4_ASYM: e = launch_a8_f<UQ_INT4_ASYM>(a, xq, sxs, sxl, Kp, grid, st); break;
        case UQ_INT8_SYM: e = launch_a8_f<UQ_INT8_SYM>(a, xq, sxs, sxl, Kp, grid, st); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess || a.cta_rows) return e;
    return launch_gemv_second_pass(a, grid, st);
}

}  // namespace uq
