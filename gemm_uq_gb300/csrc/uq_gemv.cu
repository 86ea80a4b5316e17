// uq_gemv.cu -- dispatch of the small-M GEMV over formats (kernels instantiated in uq_gemv_*.cu).
#include "uq_gemv.cuh"

namespace uq {

extern template cudaError_t launch_gemv_fmt<UQ_INT4_SYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_INT4_ASYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_INT8_SYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_INT2_ASYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_NF4>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_K4>(const GemvArgs&, int, cudaStream_t);

size_t gemv_smem_bytes(int fmt, int K, int group, int M) { return gemv_smem_bytes_impl(fmt, K, group, M); }
int gemv_warps(int fmt) { return gemv_warps_impl(fmt); }
int gemv_grid(GemvArgs& a, int fmt, int sms) {
    a.cta_rows = 0;
    if (!gemv_is_mma(fmt)) return (a.P + GEMV_WARPS - 1) / GEMV_WARPS;
    // Whole row blocks per CTA need no second pass; take them when no warp gets more tiles than
    // under the stream-K split and either the busiest CTA streams at most ~6 % more bytes than the
    // average one (bandwidth-bound shapes) or no warp has more than one tile (latency-bound ones).
    const int W = gemv_warps(fmt);
    const int G = a.NB < sms ? a.NB : sms;
    const long long rbs = (a.NB + G - 1) / G;
    const long long per_warp_rows = (rbs * a.KB + W - 1) / W;
    const long long per_warp_split = (a.T + a.P - 1) / a.P;
    const bool even = rbs * G * 100 <= (long long)a.NB * 106;
    if (G > 0 && per_warp_rows <= per_warp_split && (even || per_warp_rows <= 1)) {
        a.cta_rows = 1;
        return G;
    }
    return a.P < sms ? a.P : sms;
}
size_t gemv_partials_floats(int P, int M) { return gemv_partials_floats_impl(P, M); }

// Second pass of the mma GEMV's split-K: for every row block that several workers share, sum their
// partials in worker order (fixed, so results are bit-reproducible) and store y.  Launched right
// after the GEMV with programmatic stream serialization: it becomes resident early and its
// griddepcontrol.wait returns once the GEMV grid has finished and its stores are visible, so the
// GEMV itself needs no fence, ticket or waiting between workers.
__global__ void __launch_bounds__(256) gemv_split_reduce(const GemvArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int M = a.M, KB = a.KB;
    const long long total = (long long)a.NB * RB * M;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const bool e32 = total < (1ll << 31);
        const int nb = e32 ? (int)((unsigned)e / (unsigned)(RB * M)) : (int)(e / (RB * M));
        const int rm = e32 ? (int)((unsigned)e % (unsigned)(RB * M)) : (int)(e % (RB * M));   // r * M + m
        const int n = nb * RB + rm / M, m = rm % M;
        if (n >= a.N) continue;
        const long long tf = (long long)nb * KB;
        // worker ranges: 32-bit arithmetic when T * (P + 1) fits (every practical shape)
        const bool small = a.T * (long long)(a.P + 1) < (1ll << 31);
        int wf, wl;
        if (small) {
            const unsigned T = (unsigned)a.T, P = (unsigned)a.P, t = (unsigned)tf;
            wf = (int)(((t + 1) * P - 1) / T);
            wl = (int)(((t + KB) * P - 1) / T);
        } else {
            wf = worker_of(tf, a.T, a.P);
            wl = worker_of(tf + KB - 1, a.T, a.P);
        }
        if (wf == wl) continue;                            // one worker covered it and stored y
        float sum = 0.f;
        for (int w2 = wf; w2 <= wl; ++w2) {
            const long long b2 = small ? (long long)((unsigned)w2 * (unsigned)a.T / (unsigned)a.P)
                                       : range_begin(w2, a.T, a.P);
            const int nb2 = small ? (int)((unsigned)b2 / (unsigned)KB) : (int)(b2 / KB);
            const int slot2 = 2 * w2 + (nb == nb2 ? 0 : 1);
            sum += a.partials[(long long)slot2 * RB * M + rm];
        }
        a.y[(long long)m * a.ldy + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
    }
}

static cudaError_t launch_split_reduce(const GemvArgs& a, int sms, cudaStream_t st) {
    const long long total = (long long)a.NB * RB * a.M;
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
    if (e != cudaSuccess || !gemv_is_mma(fmt) || a.cta_rows) return e;
    // the mma kernel leaves row blocks shared between workers as partial sums (grid = its CTAs,
    // one per SM at most, so it is also the SM count bound for the reduce grid)
    return launch_split_reduce(a, grid, st);
}

}  // namespace uq
