// uq_gemm_mma.cu -- batched decode (9 <= M <= 64 activation rows) on mma.sync for the 4-bit and
// 2-bit formats (INT4_SYM, INT4_ASYM, INT2_ASYM, K4), sm_103a.
//
// "Ultra LLM Engine", section "Fused Kernels": the dequantized-weight GEMM of batched decode.  The
// packed weights are still streamed from HBM once; what changes from the GEMV is the reuse of each
// unpacked A fragment (16 weight rows x 16 k) for all M/8 column blocks of x:
//
//  * CTA = 8 warps over one row group (8 row blocks of 16 rows = 128 weight rows) and one of KS
//    contiguous ranges of its k units (unit = 4 chunks of the packed plane: 256 codes of 4-bit, 512
//    of 2-bit, 2 KB per 16-row block).  Warp w owns row block 8 rg + w for the whole range and
//    accumulates its 16 rows x 8 NB8 columns in registers, so warps never wait for each other.
//  * Each warp streams its units through a ring of its own (MMA_GEMM_STAGES buffers, per-lane
//    16-byte cp.async of the codes and 4-byte copies of the unit's scales / zero points / K4
//    record, one cp.async group per unit), requested before the wait for the previous kernel on
//    the stream since the weights are constant.
//  * A fragment: the exact integer (q - z) in bf16 (lop3 magic 128 + q, then sub.rn.bf16x2 of
//    128 + z; K4: q), so no sums of x are needed for the zero points.  B fragments come straight
//    from x in global memory through L1: the CTA's 8 warps walk the same k units at the same time,
//    so each x line is fetched into L1 once per CTA and unit.
//  * Per group: for each column block, the group's blocks as two mma chains, then y += s * D
//    (K4: d*sc_j * D - dmin*m_j * sum x, the column sums of x per 32-k sub-block from a pre-kernel).
//  * KS = 1: y is stored directly.  KS > 1: each CTA stores its partial sums [split][row][m] and a
//    second launch adds the splits in order (deterministic).
#include "uq_gemv.cuh"

namespace uq {

namespace {

constexpr int MMA_GEMM_WARPS = 8;
constexpr int MMA_GEMM_STAGES = 4;

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// A unit's staging buffer: 2 KB of codes, then per row MW words of metadata: the words covering the
// unit's scales (K4: its 16-byte record), then those covering its zero points.
template <int FMT, int GB> struct GemmUnit {
    static constexpr int UK = 4 * fmt_kc(FMT);                      // codes per unit row
    static constexpr int GS = GB * 16;
    static constexpr int GPU = UK / GS;                             // scaling groups per unit row
    static constexpr int SW = (FMT == UQ_K4) ? 4 : (2 * GPU + 5) / 4;
    static constexpr int ZW = (FMT == UQ_INT4_ASYM) ? ((GPU + 2) / 2 + 6) / 4
                            : ((FMT == UQ_INT2_ASYM) ? (2 * GPU + 5) / 4 : 0);
    static constexpr int MW = SW + ZW;
    static constexpr int STAGE = 4 * CHUNK + (RB * MW * 4 + 15) / 16 * 16;
};

template <int FMT, int GB, int NB8>
__global__ void __launch_bounds__(MMA_GEMM_WARPS * 32, 2) gemm_mma_kernel(const GemmArgs a) {
    using F = GemvFmt<FMT>;
    using U = GemmUnit<FMT, GB>;
    constexpr int S = MMA_GEMM_STAGES, KC = fmt_kc(FMT), UK = U::UK, GPU = U::GPU, MW = U::MW, SW = U::SW;
    constexpr int BPCH = F::BPC;                                    // 16-k blocks per chunk
    constexpr int WPG = (FMT == UQ_INT2_ASYM) ? GB / 2 : GB;        // code words per lane per group
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int rg = blockIdx.x / a.KS, ks = blockIdx.x % a.KS;
    const int nb = rg * MMA_GEMM_WARPS + warp;                      // this warp's row block
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (nb >= a.NB) return;                                         // past the last row block
    const int u0 = (int)((long long)ks * a.UB / a.KS), u1 = (int)((long long)(ks + 1) * a.UB / a.KS);
    const int nu = u1 - u0;
    const Layout L(a.N, a.K, FMT);
    const int G = a.K / a.group, ZB = (G + 1) >> 1, S4 = a.K / 256;
    const int G_all = a.K / U::GS;                                  // scaling groups per row
    const int n0 = nb * RB;
    const int rows = (a.N - n0) < RB ? (a.N - n0) : RB;
    const uint8_t* wrow = a.wq + (long long)nb * RB * L.rowbytes;
    uint8_t* ring = smem + (size_t)warp * S * U::STAGE;

    // unit u's codes (the chunks inside the padded row) and metadata into buffer st
    auto issue = [&](int u, uint8_t* st) {
        const int left = (L.Kp - u * UK) / KC;
        const int nch = left < 4 ? left : 4;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (q < nch) cp_async16(st + q * CHUNK + lane * 16, wrow + (long long)u * (4 * CHUNK) + q * CHUNK + lane * 16);
        uint32_t* md = reinterpret_cast<uint32_t*>(st + 4 * CHUNK);
        if constexpr (FMT == UQ_K4) {
            if (lane < rows) cp_async16(md + lane * MW, a.scales + ((long long)(n0 + lane) * S4 + u) * 16);
        } else {
            const int gi0 = u * GPU;
            const int gc = (G - gi0) < GPU ? (G - gi0) : GPU;
            const long long send = (long long)a.N * G * 2;
            for (int e = lane; e < rows * MW; e += 32) {
                const int r = e / MW, j = e % MW;
                const long long n = n0 + r;
                if (j < SW) {
                    stage_words(md + r * MW, a.scales, (n * G + gi0) * 2, gc * 2, send, j);
                } else if constexpr (FMT == UQ_INT4_ASYM) {
                    stage_words(md + r * MW + SW, a.zc, n * ZB + (gi0 >> 1), ((gi0 & 1) + gc + 1) >> 1,
                                (long long)a.N * ZB, j - SW);
                } else if constexpr (FMT == UQ_INT2_ASYM) {
                    stage_words(md + r * MW + SW, a.zc, (n * G + gi0) * 2, gc * 2, send, j - SW);
                }
            }
        }
        cp_async_commit_group();
    };

    // the weights and their metadata are constant: the first units are requested before the wait
    // for the previous kernel (which may write x, the column sums and the partial sums)
#pragma unroll
    for (int s = 0; s < S; ++s) {
        if (s < nu) issue(u0 + s, ring + s * U::STAGE);
        else cp_async_commit_group();                               // one group per slot
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    float acc[NB8][4];
#pragma unroll
    for (int cb = 0; cb < NB8; ++cb)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[cb][e] = 0.f;
    // this lane's x row of each column block (rows past M repeat the last one; their columns are
    // never stored)
    int xo[NB8];                                                    // element offsets (M x ldx fits 32 bits)
#pragma unroll
    for (int cb = 0; cb < NB8; ++cb) {
        const int m = cb * 8 + g < a.M ? cb * 8 + g : a.M - 1;
        xo[cb] = m * a.ldx + 4 * c;
    }

    int s = 0;
    for (int i = 0; i < nu; ++i) {
        cp_async_wait_group<S - 1>();                               // unit i's copies have landed
        __syncwarp();
        const uint8_t* st = ring + s * U::STAGE;
        const int u = u0 + i;
        const uint8_t* m0 = st + 4 * CHUNK + g * (MW * 4);          // metadata of rows g and g + 8
        const uint8_t* m1 = m0 + 8 * (MW * 4);
        const unsigned f0 = (unsigned)(n0 + g) * (unsigned)G + (unsigned)(u * GPU);   // low bits only
        const unsigned f1 = f0 + 8u * (unsigned)G;
#pragma unroll 1
        for (int gg = 0; gg < GPU; ++gg) {
            const int gi = u * GPU + gg;
            if (gi >= G_all) break;                                 // groups past K (warp-uniform)
            // the lane's code words of the group
            uint32_t wv[WPG];
            {
                const int blk = gg * GB;
                const uint8_t* cp = st + (blk / BPCH) * CHUNK + lane * 16 + ((blk % BPCH) * WPG / GB) * 4;
                if constexpr (WPG == 8) {
                    const uint4 v0 = *reinterpret_cast<const uint4*>(cp);
                    const uint4 v1 = *reinterpret_cast<const uint4*>(cp + CHUNK);
                    wv[0] = v0.x; wv[1] = v0.y; wv[2] = v0.z; wv[3] = v0.w;
                    wv[4] = v1.x; wv[5] = v1.y; wv[6] = v1.z; wv[7] = v1.w;
                } else if constexpr (WPG == 4) {
                    const uint4 v = *reinterpret_cast<const uint4*>(cp);
                    wv[0] = v.x; wv[1] = v.y; wv[2] = v.z; wv[3] = v.w;
                } else if constexpr (WPG == 2) {
                    const uint2 v = *reinterpret_cast<const uint2*>(cp);
                    wv[0] = v.x; wv[1] = v.y;
                } else {
                    wv[0] = *reinterpret_cast<const uint32_t*>(cp);
                }
            }
            // rows g and g + 8: scale (K4: d*sc and dmin*m of the sub-block) and the bf16 pair 128 + z
            float sc[2], dm[2] = {0.f, 0.f};
            uint32_t zz[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint8_t* mr = j ? m1 : m0;
                const unsigned f = j ? f1 : f0;
                if constexpr (FMT == UQ_K4) {
                    const uint4 rec = *reinterpret_cast<const uint4*>(mr);
                    const uint64_t sc48 = (uint64_t)rec.y | ((uint64_t)(rec.z & 0xFFFFu) << 32);
                    const uint64_t m48 = (uint64_t)(rec.z >> 16) | ((uint64_t)rec.w << 16);
                    sc[j] = half_bits_f32((uint16_t)(rec.x & 0xFFFF)) * (float)((sc48 >> (6 * gg)) & 63);
                    dm[j] = half_bits_f32((uint16_t)(rec.x >> 16)) * (float)((m48 >> (6 * gg)) & 63);
                    zz[j] = 0x43004300u;                            // A = q
                } else {
                    sc[j] = half_bits_f32(reinterpret_cast<const uint16_t*>(mr + 2 * (f & 1u))[gg]);
                    uint32_t z;
                    if constexpr (FMT == UQ_INT4_SYM) {
                        z = 8u;                                     // codes are stored biased by 8
                    } else if constexpr (FMT == UQ_INT4_ASYM) {
                        const unsigned zb0 = (unsigned)(n0 + g + 8 * j) * (unsigned)ZB + (unsigned)((u * GPU) >> 1);
                        const uint32_t b = mr[SW * 4 + (zb0 & 3u) + (gg >> 1)];
                        z = (gg & 1) ? (b >> 4) : (b & 15u);
                    } else {
                        z = (uint32_t)half_bits_f32(reinterpret_cast<const uint16_t*>(mr + SW * 4 + 2 * (f & 1u))[gg]);
                    }
                    zz[j] = (0x4300u | z) * 0x00010001u;            // bf16 pair (128 + z, 128 + z)
                }
            }
            // A fragments: exact (q - z) bf16 pairs; registers 0, 2 hold row g, 1, 3 row g + 8
            uint32_t af[GB][4];
#pragma unroll
            for (int j = 0; j < GB; ++j) {
                uint32_t a0, a1, a2, a3;
                if constexpr (FMT == UQ_INT2_ASYM) {
                    const uint32_t wd = wv[j >> 1];
                    if (j & 1) {
                        a0 = crumb_pair_lop3<4>(wd); a1 = crumb_pair_lop3<5>(wd);
                        a2 = crumb_pair_lop3<6>(wd); a3 = crumb_pair_lop3<7>(wd);
                    } else {
                        a0 = crumb_pair_lop3<0>(wd); a1 = crumb_pair_lop3<1>(wd);
                        a2 = crumb_pair_lop3<2>(wd); a3 = crumb_pair_lop3<3>(wd);
                    }
                } else {
                    const uint32_t wd = wv[j];
                    a0 = nib_pair_lop3<0>(wd); a1 = nib_pair_lop3<1>(wd);
                    a2 = nib_pair_lop3<2>(wd); a3 = nib_pair_lop3<3>(wd);
                }
                af[j][0] = bf16x2_sub(a0, zz[0]);
                af[j][1] = bf16x2_sub(a1, zz[1]);
                af[j][2] = bf16x2_sub(a2, zz[0]);
                af[j][3] = bf16x2_sub(a3, zz[1]);
            }
            const int kg = u * UK + gg * U::GS;                     // the group's first k
#pragma unroll
            for (int cb = 0; cb < NB8; ++cb) {
                float dd[2][4];
#pragma unroll
                for (int j = 0; j < GB; ++j) {
                    const uint2 bv = ldg_nc_v2(a.x + (xo[cb] + kg + j * 16));
                    if (j < 2) mma_bf16_zero(dd[j & 1], af[j][0], af[j][1], af[j][2], af[j][3], bv.x, bv.y);
                    else mma_bf16(dd[j & 1], af[j][0], af[j][1], af[j][2], af[j][3], bv.x, bv.y);
                }
                if constexpr (FMT == UQ_K4) {
                    const int cm = cb * 8 + 2 * c;
                    const float2 sxv = *reinterpret_cast<const float2*>(a.sx + (long long)(kg / 32) * a.Mpad + cm);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        acc[cb][2 * j] = fmaf(sc[j], dd[0][2 * j] + dd[1][2 * j], fmaf(-dm[j], sxv.x, acc[cb][2 * j]));
                        acc[cb][2 * j + 1] = fmaf(sc[j], dd[0][2 * j + 1] + dd[1][2 * j + 1], fmaf(-dm[j], sxv.y, acc[cb][2 * j + 1]));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        acc[cb][2 * j] = fmaf(sc[j], dd[0][2 * j] + dd[1][2 * j], acc[cb][2 * j]);
                        acc[cb][2 * j + 1] = fmaf(sc[j], dd[0][2 * j + 1] + dd[1][2 * j + 1], acc[cb][2 * j + 1]);
                    }
                }
            }
        }
        __syncwarp();                                               // every lane is done with the buffer
        if (i + S < nu) issue(u0 + i + S, ring + s * U::STAGE);
        else cp_async_commit_group();
        if (++s == S) s = 0;
    }
    cp_async_wait_group<0>();

    // rows g, g + 8; columns cb * 8 + 2c + e
#pragma unroll
    for (int cb = 0; cb < NB8; ++cb)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int m = cb * 8 + 2 * c + e, r = g + 8 * j;
                if (m >= a.M || r >= rows) continue;
                if (a.KS == 1) store_out(a, m, n0 + r, acc[cb][2 * j + e]);
                else a.partials[((long long)ks * a.NB * RB + n0 + r) * a.M + m] = acc[cb][2 * j + e];
            }
}

template <int FMT, int GB, int NB8>
cudaError_t launch_gemm_mma_t(const GemmArgs& a, cudaStream_t st) {
    static bool configured[64] = {};
    const size_t smem = (size_t)MMA_GEMM_WARPS * MMA_GEMM_STAGES * GemmUnit<FMT, GB>::STAGE;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gemm_mma_kernel<FMT, GB, NB8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int grid = ((a.NB + MMA_GEMM_WARPS - 1) / MMA_GEMM_WARPS) * a.KS;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(MMA_GEMM_WARPS * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = launch_overlap() ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, gemm_mma_kernel<FMT, GB, NB8>, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int FMT, int GB>
cudaError_t launch_gemm_mma_nb(const GemmArgs& a, cudaStream_t st) {
    if (a.M <= 16) return launch_gemm_mma_t<FMT, GB, 2>(a, st);
    if (a.M <= 32) return launch_gemm_mma_t<FMT, GB, 4>(a, st);
    return launch_gemm_mma_t<FMT, GB, 8>(a, st);
}

template <int FMT>
cudaError_t launch_gemm_mma_fmt(const GemmArgs& a, cudaStream_t st) {
    if constexpr (FMT == UQ_K4) {
        return launch_gemm_mma_nb<FMT, 2>(a, st);
    } else {
        switch (a.group) {
            case 32: return launch_gemm_mma_nb<FMT, 2>(a, st);
            case 64: return launch_gemm_mma_nb<FMT, 4>(a, st);
            case 128: return launch_gemm_mma_nb<FMT, 8>(a, st);
            default: return cudaErrorInvalidValue;
        }
    }
}

}  // namespace

int gemm_mma_units(int fmt, int K) {
    const int kc = fmt_kc(fmt), uk = 4 * kc;
    const int Kp = (K + kc - 1) / kc * kc;
    return (Kp + uk - 1) / uk;
}

int gemm_mma_splits(int NB, int UB, int sms) {
    // k splits per row group: the fewest that minimise the units of the busiest SM, counted as
    // (CTAs the SM runs) x (units per CTA) with the CTAs spread evenly over the SMs
    const long long RG = (NB + MMA_GEMM_WARPS - 1) / MMA_GEMM_WARPS;
    int best = 1;
    long long best_load = -1;
    for (int ks = 1; ks <= UB && ks <= 64; ++ks) {
        const long long ctas = RG * ks;
        const long long load = (ctas + sms - 1) / sms * ((UB + ks - 1) / ks);
        if (best_load < 0 || load < best_load) {
            best_load = load;
            best = ks;
        }
    }
    return best;
}

cudaError_t launch_gemm_mma(int fmt, const GemmArgs& a, int sms, cudaStream_t st) {
    cudaError_t e;
    switch (fmt) {
        case UQ_INT4_SYM: e = launch_gemm_mma_fmt<UQ_INT4_SYM>(a, st); break;
        case UQ_INT4_ASYM: e = launch_gemm_mma_fmt<UQ_INT4_ASYM>(a, st); break;
        case UQ_INT2_ASYM: e = launch_gemm_mma_fmt<UQ_INT2_ASYM>(a, st); break;
        case UQ_K4: e = launch_gemm_mma_fmt<UQ_K4>(a, st); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess || a.KS == 1) return e;
    // the splits' partial sums [KS][rows][M], added in split order by the GEMV's second pass
    GemvArgs r = {};
    r.M = a.M; r.N = a.N; r.NB = a.NB; r.KB = a.KS;
    r.partials = a.partials;
    r.y = a.y; r.ldy = a.ldy;
    r.out32 = a.out32; r.gate32 = a.gate32;
    return launch_gemv_second_pass(r, sms, st);
}

}  // namespace uq
