// uq_gemv.cu -- dispatch of the small-M GEMV over formats (kernels instantiated in uq_gemv_*.cu).
#include "uq_gemv.cuh"

namespace uq {

extern template cudaError_t launch_gemv_fmt<UQ_INT4_SYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_INT4_ASYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_INT8_SYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_INT2_ASYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_NF4>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_K4>(const GemvArgs&, int, cudaStream_t);

// Per-warp rings (gemv_warp_kernel): W warps per CTA, cps CTAs per SM.  Whole row
// blocks per CTA need no second pass; take them when no warp gets more tiles than under the
// stream-K split (or one more, from 3 tiles a warp up: measured on the 8B down projection,
// 4096 x 14336, 4 tiles a warp and no second pass beat 3 and the second pass, 3221 against 3056
// GB/s on the M = 1 sweep) and either the busiest CTA streams at most ~6 % more bytes than the
// average one (bandwidth-bound shapes) or no warp has more than one tile (latency-bound ones).
// (gated: the units CTAs own are gate/up pairs of row blocks)
static int plan_warp_rings(GemvArgs& a, int sms, int W, int cps, int tpw) {
    const int WU = a.gated ? 2 : 1;
    const int NBU = a.NB / WU;
    const long long P = (long long)sms * cps * W;
    a.P = (int)(P < a.T ? P : a.T);
    const int slots = sms * cps;                                       // CTAs resident at once
    const int G = NBU < slots ? NBU : slots;
    const long long rbs = G > 0 ? (NBU + G - 1) / G : 0;
    const long long per_warp_rows = (rbs * WU * a.KB + W - 1) / W;
    const long long per_warp_split = (a.T + a.P - 1) / a.P;
    const bool even = rbs * G * 100 <= (long long)NBU * 106;
    const long long slack = per_warp_split >= 3 ? 1 : 0;
    if (G > 0 && per_warp_rows <= tpw && per_warp_rows <= per_warp_split + slack && (even || per_warp_rows <= 1)) {
        a.cta_rows = 1;
        return G;
    }
    return a.P < slots ? a.P : slots;
}

int gemv_plan(GemvArgs& a, int fmt, int sms) {
    a.cta_rows = 0;
    const int WU = a.gated ? 2 : 1;
    const int NBU = a.NB / WU;
    if (!a.a8 && gemv_warp_route(fmt, a.M))
        return plan_warp_rings(a, sms, WarpCfg<UQ_INT4_ASYM>::WARPS, WARP_CTAS_PER_SM, WARP_TPW);
    // mma GEMV: one CTA per SM, its work (pairs of k tiles) shared by MMA_CW compute warps.  Whole
    // row blocks per CTA (a.cta_rows = the most tiles a CTA gets) need no second pass; take them
    // when every compute warp has one tile at most (latency-bound shapes), or when no CTA gets more
    // tiles than under the stream-K split and the busiest CTA streams at most ~6 % more bytes than
    // the average one, or when it gets at most 2 pairs of tiles more and all of x still fits in
    // shared memory beside the ring (measured: the M = 2 sweep 2527 -> 2657 GB/s from its 4096 x
    // 14336 down projection, W4A8 at M = 1 2036 -> 2101, INT2 g64 8192^2 at M = 1 1886 -> 2032,
    // NF4 g64 1723 -> 1878; with x read through L1 instead, M = 8 lost 20 %).
    const int slots = sms;
    const long long KB2 = (a.KB + 1) / 2;
    const long long P2 = (long long)a.NB * KB2;                        // pairs of k tiles
    if (P2 >= (1LL << 31)) return 0;                                   // the kernel splits in 32-bit arithmetic
    const int grid_split = (int)(P2 < slots ? P2 : slots);
    const long long per_cta_split = 2 * ((P2 + grid_split - 1) / grid_split);
    const int G = NBU < slots ? NBU : slots;
    int grid = grid_split;
    if (G > 0) {
        const long long rbs = (NBU + G - 1) / G;
        const long long tc = rbs * WU * 2 * KB2;
        const bool even = rbs * G * 100 <= (long long)NBU * 106;
        bool near = false;
        if (tc <= MMA_TPC && tc > per_cta_split && tc <= per_cta_split + 4) {
            const int sxg_rows = gemv_mma_sx_groups(fmt, a.group, a.NB, a.KB, G, (int)tc);
            near = gemv_mma_smem(fmt, a.K, a.group, a.M, sxg_rows, (int)tc, MMA_X_WHOLE, a.a8 ? 1 : 2).S2 >=
                   MMA_CW / 2 + 2;
        }
        if (tc <= MMA_TPC && (tc <= MMA_CW || (tc <= per_cta_split && even) || near)) {
            a.cta_rows = (int)tc;
            grid = G;
        }
    }
    a.P = grid;
    const int sxg = gemv_mma_sx_groups(fmt, a.group, a.NB, a.KB, grid, a.cta_rows);
    if (gemv_mma_smem(fmt, a.K, a.group, a.M, sxg, a.cta_rows, MMA_X_GLOBAL).S2 < MMA_CW / 2 + 2) {
        a.cta_rows = 0;
        return 0;
    }
    return grid;
}

size_t gemv_partials_floats(int fmt, const GemvArgs& a) {
    // one 16-row slot per tile (k-major tiles, summed over k by the second pass)
    (void)fmt;
    return a.cta_rows ? 0 : (size_t)a.T * RB * a.M;
}
bool gemv_uses_tickets(int fmt, const GemvArgs& a) {
    (void)fmt;
    (void)a;
    return false;                       // every GEMV sums shared row blocks in its second pass
}
int gemv_launches(int fmt, const GemvArgs& a) {
    (void)fmt;
    return a.cta_rows ? 1 : 2;
}

// Second pass of the mma GEMV when workers split the matrix's tiles (k-major, so every tile's
// partial sums have a slot of their own): y[m][n] = the sum over k tiles, in k order (fixed, so
// results are bit-reproducible).  Launched right after the GEMV with programmatic stream
// serialization: it becomes resident early and its griddepcontrol.wait returns once the GEMV grid
// has finished and its stores are visible, so the GEMV itself needs no fence or ticket.
// Gated (a.gated): work row block 2j is gate row block j, 2j + 1 the up one; h = silu(g) * u.
__global__ void __launch_bounds__(256) gemv_split_reduce(const GemvArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int M = a.M, KB = a.KB, RM = RB * M;
    const int WU = a.gated ? 2 : 1;
    const long long total = (long long)(a.NB / WU) * RM;
    const long long kstride = (long long)a.NB * RM;                 // floats between k tiles
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int nb = (int)(e / RM), rm = (int)(e % RM);           // rm = r * M + m
        const int n = nb * RB + rm / M, m = rm % M;
        if (n >= a.N) continue;
        const float* p = a.partials + (long long)nb * WU * RM + rm; // k tile 0 of (work row block, r, m)
        float sum = 0.f;
        for (int kb = 0; kb < KB; ++kb) sum += p[kb * kstride];
        if (a.gated) {
            float usum = 0.f;
            for (int kb = 0; kb < KB; ++kb) usum += p[kb * kstride + RM];
            a.y[(long long)m * a.ldy + n] = __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul(sum, usum)));
        } else {
            store_out(a, m, n, sum);
        }
    }
}

cudaError_t launch_gemv_second_pass(const GemvArgs& a, int sms, cudaStream_t st) {
    const long long total = (long long)(a.gated ? a.NB / 2 : a.NB) * RB * a.M;
    long long blocks = (total + 255) / 256;
    if (blocks > 4LL * sms) blocks = 4LL * sms;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_split_reduce, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_gemv(int fmt, const GemvArgs& a, int grid, cudaStream_t st) {
    cudaError_t e;
    switch (fmt) {
        case UQ_INT4_SYM: e = launch_gemv_fmt<UQ_INT4_SYM>(a, grid, st); break;
        case UQ_INT4_ASYM: e = launch_gemv_fmt<UQ_INT4_ASYM>(a, grid, st); break;
        case UQ_INT8_SYM: e = launch_gemv_fmt<UQ_INT8_SYM>(a, grid, st); break;
        case UQ_INT2_ASYM: e = launch_gemv_fmt<UQ_INT2_ASYM>(a, grid, st); break;
        case UQ_NF4: e = launch_gemv_fmt<UQ_NF4>(a, grid, st); break;
        case UQ_K4: e = launch_gemv_fmt<UQ_K4>(a, grid, st); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess || a.cta_rows) return e;
    // the mma kernel leaves row blocks shared between workers as partial sums (grid = its CTAs,
    // one per SM at most, so it is also the SM count bound for the reduce grid)
    return launch_gemv_second_pass(a, grid, st);
}

}  // namespace uq
