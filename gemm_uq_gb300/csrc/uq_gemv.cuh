// uq_gemv.cuh -- small-M (M <= 8) fused dequantize + GEMV/GEMM on CUDA cores, sm_103a.
//
// "Ultra LLM Engine", section "Fused Kernels": dequantized-weight GEMV for single-token
// decode and GEMM for batched decode.  Decode is bound by streaming the packed weights
// from HBM once, so the kernel is organised around that stream:
//
//  * Work is the list of tiles (8 rows x 512 bytes of codes) in row-block-major order.
//    Every warp is an independent worker that owns a contiguous, equal share of that list
//    (a "stream-K" split: balanced over 152 SMs x 8 warps whatever N and K are).
//  * Each warp keeps GEMV_STAGES tiles in flight in a warp-private ring in shared memory.
//    One stage holds a tile's codes (one 1-D bulk async copy, cp.async.bulk, issued by lane 0)
//    AND the tile's scales / zero points / K4 records (4- or 16-byte cp.async copies issued by
//    all lanes); both complete on the stage's mbarrier (expect_tx for the bulk bytes, one
//    cp.async.mbarrier.arrive.noinc per lane), so a tile's metadata is prefetched as deep
//    as its weights and the consumer never waits on a global load.
//  * x is copied once per CTA into shared memory (in lane-chunk order, so the per-tile reads
//    are conflict-free 16-byte loads) together with the per-chunk sums of x; the prologue
//    runs while the first weight tiles are already in flight.
//  * Lane l owns the 16-byte column chunk l of every tile row (32 INT4 codes).  Codes are
//    unpacked with the magic-exponent trick (bf16 0x4300 | code = 128 + code) and multiplied-
//    accumulated with fma.rn.f32.bf16 (fp32 accumulate of exact bf16 products).  The +128
//    offset and the zero point are removed once per group:
//        sum x*(q - z) = sum x*(128 + q) - (128 + z) * sum x.
//  * A row block whose k range is split between workers is finished by a deterministic
//    second pass: each contributor stores its fp32 partial sums, takes a ticket, and the
//    last one sums the partials in worker order (fixed, so results are bit-reproducible)
//    and writes y.  No worker ever waits for another.
#pragma once
#include "uq_kernels.h"

namespace uq {

// per-format staging constants
template <int FMT> struct GemvFmt {
    static constexpr int KT = fmt_kt(FMT);
    static constexpr int CPL = fmt_cpl(FMT);
    static constexpr int GT_MAX = KT / 32;                         // groups per tile row at group 32
    // 32-bit words of metadata staged per tile row: scales (+1 for a misaligned start), zeros
    static constexpr int SW = (FMT == UQ_K4) ? 16 : GT_MAX / 2 + 1;
    static constexpr int ZW = (FMT == UQ_INT4_ASYM) ? GT_MAX / 8 + 1 : (FMT == UQ_INT2_ASYM ? GT_MAX / 2 + 1 : 0);
    static constexpr int MW = SW + ZW;
    static constexpr int META_BYTES = (RB * MW * 4 + 15) / 16 * 16;
    static constexpr int STAGE_BYTES = TILE_BYTES + META_BYTES;
    static constexpr int STAGES = (FMT == UQ_INT2_ASYM) ? 3 : 4;
    static constexpr bool NEEDS_SX = (FMT != UQ_INT8_SYM && FMT != UQ_NF4);
    static constexpr int HALVES = (FMT == UQ_INT2_ASYM) ? 2 : 1;
};

// shared-memory plan; identical on host and device
struct GemvSmem {
    size_t ring, bars, lut, sx, x, total;
};
__host__ __device__ inline GemvSmem gemv_smem_plan(int fmt, int K, int M, bool x_in_smem) {
    int stage = 0, stages = 0, cpl = fmt_cpl(fmt), kt = fmt_kt(fmt);
    switch (fmt) {
        case UQ_INT4_SYM: stage = GemvFmt<UQ_INT4_SYM>::STAGE_BYTES; stages = GemvFmt<UQ_INT4_SYM>::STAGES; break;
        case UQ_INT4_ASYM: stage = GemvFmt<UQ_INT4_ASYM>::STAGE_BYTES; stages = GemvFmt<UQ_INT4_ASYM>::STAGES; break;
        case UQ_INT8_SYM: stage = GemvFmt<UQ_INT8_SYM>::STAGE_BYTES; stages = GemvFmt<UQ_INT8_SYM>::STAGES; break;
        case UQ_INT2_ASYM: stage = GemvFmt<UQ_INT2_ASYM>::STAGE_BYTES; stages = GemvFmt<UQ_INT2_ASYM>::STAGES; break;
        case UQ_NF4: stage = GemvFmt<UQ_NF4>::STAGE_BYTES; stages = GemvFmt<UQ_NF4>::STAGES; break;
        default: stage = GemvFmt<UQ_K4>::STAGE_BYTES; stages = GemvFmt<UQ_K4>::STAGES; break;
    }
    const size_t kbt = (size_t)(K + kt - 1) / kt;
    const bool needs_sx = (fmt != UQ_INT8_SYM && fmt != UQ_NF4);
    GemvSmem p;
    p.ring = 0;
    p.bars = (size_t)GEMV_WARPS * stages * stage;
    p.lut = p.bars + (size_t)GEMV_WARPS * stages * 8;
    p.sx = p.lut + 64;
    p.x = p.sx + (needs_sx ? kbt * (fmt == UQ_INT2_ASYM ? 2 : 1) * M * 32 * 4 : 0);
    p.x = (p.x + 15) / 16 * 16;
    p.total = p.x + (x_in_smem ? kbt * M * (cpl / 8) * 32 * 16 : 0);
    return p;
}

namespace {

__device__ __forceinline__ long long range_begin(int w, long long T, int P) { return (long long)w * T / P; }
__device__ __forceinline__ int worker_of(long long t, long long T, int P) {
    return (int)(((t + 1) * (long long)P - 1) / T);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(bar)) : "memory");
}

// Copy the 4-byte-aligned words covering bytes [lo, lo + len) of `base` into dst (word 0 holds
// byte lo & ~3).  A word that would reach past `end` (the array's end) is assembled from plain
// byte loads instead, so nothing outside the caller's buffer is read.
__device__ __forceinline__ void stage_words(uint32_t* dst, const uint8_t* base, long long lo, int len,
                                            long long end, int j) {
    const long long w0 = lo & ~3ll;
    const long long src = w0 + 4ll * j;
    if (src >= lo + len) return;
    if (src + 4 <= end) {
        cp_async4(dst + j, base + src);
    } else {
        uint32_t v = 0;
        for (int b = 0; b < 4; ++b)
            if (src + b < end) v |= (uint32_t)__ldg(base + src + b) << (8 * b);
        dst[j] = v;
    }
}

// Issue the copies of tile t into stage buffer `st` (all lanes take part).
template <int FMT>
__device__ __forceinline__ void issue_tile(const GemvArgs& a, const Layout& L, long long t, uint8_t* st,
                                           uint64_t* bar, int lane) {
    using F = GemvFmt<FMT>;
    const int nb = (int)(t / L.KB), kb = (int)(t % L.KB);
    const int rows = L.rows(nb), n0 = nb * RB;
    uint32_t* md = reinterpret_cast<uint32_t*>(st + TILE_BYTES);
    if constexpr (FMT == UQ_K4) {
        // 16-byte records: width/256 per row, 16-byte aligned
        const int recs = L.width(kb) / 256;
        for (int e = lane; e < rows * recs; e += 32) {
            const int r = e / recs, j = e % recs;
            const uint8_t* src = a.scales + ((long long)(n0 + r) * (a.K / 256) + (long long)kb * 4 + j) * 16;
            cp_async16(md + r * F::MW + 4 * j, src);
        }
    } else {
        const int G = a.K / a.group;
        const int GT = L.KT / a.group;                 // groups per full tile row
        const int gc = L.width(kb) / a.group;          // groups in this tile row
        const long long send = (long long)a.N * G * 2;
        for (int e = lane; e < rows * F::MW; e += 32) {
            const int r = e / F::MW, j = e % F::MW;
            const long long n = n0 + r;
            if (j < F::SW) {
                stage_words(md + r * F::MW, a.scales, (n * G + (long long)kb * GT) * 2, gc * 2, send, j);
            } else if constexpr (FMT == UQ_INT4_ASYM) {
                const long long ZB = (G + 1) >> 1;
                stage_words(md + r * F::MW + F::SW, a.zc, n * ZB + (long long)kb * (GT >> 1), (gc + 1) >> 1,
                            (long long)a.N * ZB, j - F::SW);
            } else if constexpr (FMT == UQ_INT2_ASYM) {
                stage_words(md + r * F::MW + F::SW, a.zc, (n * G + (long long)kb * GT) * 2, gc * 2, send, j - F::SW);
            }
        }
    }
    cp_async_arrive_noinc(bar);
    __syncwarp();
    if (lane == 0) {
        const uint32_t bytes = (uint32_t)(rows * L.slice_bytes(kb));
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(st, a.wq + L.tile_offset(nb, kb), bytes, bar);
    }
}

// per-row metadata of the lane's chunk, converted to what the accumulate step needs
struct RowMeta {
    float s;     // scale (s, a, or d*sc for K4)
    float zc;    // value subtracted per unit of sum(x): 128 + z (INT*), 136 (INT4_SYM), 128 (K4)
    float s2;    // INT2 group-32 second half: scale;  K4: dmin*m
    float zc2;   // INT2 group-32 second half: 128 + z
};

// Read row r's metadata for lane chunk starting at k0 from the staged words of tile (nb, kb).
template <int FMT>
__device__ __forceinline__ RowMeta stage_meta(const GemvArgs& a, const Layout& L, const uint8_t* st, int r, int n,
                                              int kb, int lane) {
    using F = GemvFmt<FMT>;
    const uint8_t* row = st + TILE_BYTES + r * F::MW * 4;
    RowMeta m{0.f, 0.f, 0.f, 0.f};
    if constexpr (FMT == UQ_K4) {
        const int li = lane >> 3;                  // super-block within the tile row
        const int j = lane & 7;                    // sub-block
        const uint4 rec = *reinterpret_cast<const uint4*>(row + 16 * li);
        const float d = half_bits_f32((uint16_t)(rec.x & 0xFFFF));
        const float dmin = half_bits_f32((uint16_t)(rec.x >> 16));
        const uint64_t sc48 = (uint64_t)rec.y | ((uint64_t)(rec.z & 0xFFFFu) << 32);
        const uint64_t m48 = (uint64_t)(rec.z >> 16) | ((uint64_t)rec.w << 16);
        m.s = d * (float)((sc48 >> (6 * j)) & 63);
        m.s2 = dmin * (float)((m48 >> (6 * j)) & 63);
        m.zc = 128.0f;
    } else {
        const int G = a.K / a.group, GT = L.KT / a.group;
        const int li = (lane * F::CPL) / a.group;  // first group of the chunk within the tile row
        const long long sbyte = ((long long)n * G + (long long)kb * GT) * 2;
        const uint16_t* sp = reinterpret_cast<const uint16_t*>(row + (sbyte & 3)) + li;
        m.s = half_bits_f32(sp[0]);
        if constexpr (FMT == UQ_INT4_SYM) {
            m.zc = 136.0f;
        } else if constexpr (FMT == UQ_INT4_ASYM) {
            const long long ZB = (G + 1) >> 1;
            const long long zbyte = (long long)n * ZB + (long long)kb * (GT >> 1);
            const uint32_t b = row[F::SW * 4 + (zbyte & 3) + (li >> 1)];
            // fp32 with exponent 134 and z at mantissa bits 16..19 is exactly 128 + z
            m.zc = __uint_as_float(0x43000000u | (((li & 1) ? (b >> 4) : (b & 15u)) << 16));
        } else if constexpr (FMT == UQ_INT2_ASYM) {
            const uint16_t* zp = reinterpret_cast<const uint16_t*>(row + F::SW * 4 + (sbyte & 3)) + li;
            m.zc = 128.0f + half_bits_f32(zp[0]);
            if (a.group == 32) {
                m.s2 = half_bits_f32(sp[1]);
                m.zc2 = 128.0f + half_bits_f32(zp[1]);
            }
        }
    }
    return m;
}

// One pass over the tile's rows for x rows M0 .. M0+MP-1.
template <int FMT, int M, int M0, int MP, bool XS>
__device__ __forceinline__ void tile_pass(const uint8_t* __restrict__ tile, int slice_bytes, int rows, int lane,
                                          const uint16_t* __restrict__ xg, int ldx, const uint4* __restrict__ xs,
                                          const RowMeta (&meta)[RB], float (&acc)[RB][M],
                                          const float* __restrict__ lut, bool two_groups,
                                          const float* __restrict__ sxt) {
    constexpr int CPL = fmt_cpl(FMT);
    constexpr int XU = CPL / 8;                    // 16-byte units of x per lane chunk
    auto load_x = [&](int i, int v) -> uint4 {
        if constexpr (XS) return xs[((M0 + i) * XU + v) * 32 + lane];
        else return ldg_nc_v4(xg + (long long)(M0 + i) * ldx + 8 * v);
    };
    if constexpr (FMT == UQ_INT4_SYM || FMT == UQ_INT4_ASYM || FMT == UQ_K4 || FMT == UQ_INT2_ASYM) {
        constexpr int XR = CPL / 2;                // bf16 pairs of x per lane chunk
        uint32_t xr[MP][XR];
        float sx[MP], sx2[MP];
#pragma unroll
        for (int i = 0; i < MP; ++i) {
#pragma unroll
            for (int v = 0; v < XU; ++v) {
                const uint4 q = load_x(i, v);
                xr[i][4 * v] = q.x; xr[i][4 * v + 1] = q.y; xr[i][4 * v + 2] = q.z; xr[i][4 * v + 3] = q.w;
            }
            sx[i] = sxt[(M0 + i) * 32 + lane];
            sx2[i] = 0.f;
            if constexpr (FMT == UQ_INT2_ASYM) {
                if (two_groups) sx2[i] = sxt[(M + M0 + i) * 32 + lane];
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            if (r < rows) {
                const uint4 c = *reinterpret_cast<const uint4*>(tile + r * slice_bytes + lane * 16);
                const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
                float p0[MP], p1[MP];
#pragma unroll
                for (int i = 0; i < MP; ++i) { p0[i] = 0.f; p1[i] = 0.f; }
                if constexpr (FMT == UQ_INT2_ASYM) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int p = 0; p < 8; ++p) {
                            const uint32_t t = crumb_pair_bf16(wv[j], p);
#pragma unroll
                            for (int i = 0; i < MP; ++i) {
                                if (j < 2) p0[i] = fma2_bf16(t, xr[i][8 * j + p], p0[i]);
                                else p1[i] = fma2_bf16(t, xr[i][8 * j + p], p1[i]);
                            }
                        }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            const uint32_t t = nib_pair_bf16(wv[j], p);
#pragma unroll
                            for (int i = 0; i < MP; ++i) {
                                if (j < 2) p0[i] = fma2_bf16(t, xr[i][4 * j + p], p0[i]);
                                else p1[i] = fma2_bf16(t, xr[i][4 * j + p], p1[i]);
                            }
                        }
                }
                const RowMeta& mt = meta[r];
#pragma unroll
                for (int i = 0; i < MP; ++i) {
                    float& A = acc[r][M0 + i];
                    if constexpr (FMT == UQ_INT2_ASYM) {
                        if (two_groups) {
                            A = fmaf(mt.s, fmaf(-mt.zc, sx[i], p0[i]), A);
                            A = fmaf(mt.s2, fmaf(-mt.zc2, sx2[i], p1[i]), A);
                        } else {
                            A = fmaf(mt.s, fmaf(-mt.zc, sx[i], p0[i] + p1[i]), A);
                        }
                    } else {
                        A = fmaf(mt.s, fmaf(-mt.zc, sx[i], p0[i] + p1[i]), A);
                        if constexpr (FMT == UQ_K4) A = fmaf(-mt.s2, sx[i], A);
                    }
                }
            }
        }
    } else {
        // INT8_SYM and NF4: x in fp32 registers, codes to fp32 per element
        float xf[MP][CPL];
#pragma unroll
        for (int i = 0; i < MP; ++i) {
#pragma unroll
            for (int v = 0; v < XU; ++v) {
                const uint4 q = load_x(i, v);
                const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    xf[i][8 * v + 2 * e] = bf16lo_f32(u[e]);
                    xf[i][8 * v + 2 * e + 1] = bf16hi_f32(u[e]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            if (r < rows) {
                const uint4 c = *reinterpret_cast<const uint4*>(tile + r * slice_bytes + lane * 16);
                const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
                float p0[MP], p1[MP];
#pragma unroll
                for (int i = 0; i < MP; ++i) { p0[i] = 0.f; p1[i] = 0.f; }
                if constexpr (FMT == UQ_INT8_SYM) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float q = byte_magic_f32(wv[j], e) - 8388736.0f;   // 2^23 + 128
#pragma unroll
                            for (int i = 0; i < MP; ++i) {
                                if (e & 1) p1[i] = fmaf(xf[i][4 * j + e], q, p1[i]);
                                else p0[i] = fmaf(xf[i][4 * j + e], q, p0[i]);
                            }
                        }
                } else {  // NF4: code = index into the 16-entry codebook held in shared memory
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int pos = code_bitpos(4, e);
                            const float cv = lut[(wv[j] >> pos) & 15u];
#pragma unroll
                            for (int i = 0; i < MP; ++i) {
                                if (e & 1) p1[i] = fmaf(xf[i][8 * j + e], cv, p1[i]);
                                else p0[i] = fmaf(xf[i][8 * j + e], cv, p0[i]);
                            }
                        }
                }
#pragma unroll
                for (int i = 0; i < MP; ++i) acc[r][M0 + i] = fmaf(meta[r].s, p0[i] + p1[i], acc[r][M0 + i]);
            }
        }
    }
}

template <int FMT> struct PassPlan {
    // rows of x handled per pass (register budget): INT2 and the fp32-x formats take fewer
    static constexpr int MAXP = (FMT == UQ_INT2_ASYM || FMT == UQ_NF4) ? 2 : 4;
};

template <int FMT, int M, int M0, bool XS>
__device__ __forceinline__ void tile_all_passes(const uint8_t* tile, int slice_bytes, int rows, int lane,
                                                const uint16_t* xg, int ldx, const uint4* xs,
                                                const RowMeta (&meta)[RB], float (&acc)[RB][M], const float* lut,
                                                bool two_groups, const float* sxt) {
    if constexpr (M0 < M) {
        constexpr int REM = M - M0;
        constexpr int MP = REM < PassPlan<FMT>::MAXP ? REM : PassPlan<FMT>::MAXP;
        tile_pass<FMT, M, M0, MP, XS>(tile, slice_bytes, rows, lane, xg, ldx, xs, meta, acc, lut, two_groups, sxt);
        tile_all_passes<FMT, M, M0 + MP, XS>(tile, slice_bytes, rows, lane, xg, ldx, xs, meta, acc, lut, two_groups,
                                             sxt);
    }
}

// Transposing butterfly: reduces CNT values per lane over the warp.  At each level a lane keeps
// half of its values and sends the other half to its xor partner, so every sum is formed once, in
// a fixed order; when one value is left the remaining levels are plain xor sums (commutative, so
// both partners hold identical bits).  Afterwards lane l holds the totals of value indices
// idx_out + j for j < max(1, CNT / 32) in v[j].
template <int CNT>
__device__ __forceinline__ void warp_reduce_transposed(float (&v)[CNT], int lane, int& idx_out) {
    int idx = 0;
    int half = CNT / 2;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (half >= 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < CNT / 2; ++i) {
                if (i < half) {
                    const float keep = up ? v[i + half] : v[i];
                    const float send = up ? v[i] : v[i + half];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            if (up) idx += half;
            half >>= 1;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
    idx_out = idx;
}

}  // namespace

template <int FMT, int M, bool XS>
__global__ void __launch_bounds__(GEMV_WARPS * 32, 1) gemv_kernel(const GemvArgs a) {
    using F = GemvFmt<FMT>;
    constexpr int KT = F::KT, CPL = F::CPL, S = F::STAGES;
    extern __shared__ __align__(128) uint8_t smem[];
    const GemvSmem plan = gemv_smem_plan(FMT, a.K, M, XS);
    uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + plan.bars);
    float* lut = reinterpret_cast<float*>(smem + plan.lut);
    float* sx_tab = reinterpret_cast<float*>(smem + plan.sx);
    uint4* x_tab = reinterpret_cast<uint4*>(smem + plan.x);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = blockIdx.x * GEMV_WARPS + warp;
    const bool has_work = w < a.P;
    const Layout L(a.N, a.K, FMT);
    uint8_t* ring = smem + (size_t)warp * S * F::STAGE_BYTES;
    uint64_t* bars = bars_all + warp * S;
    const long long t0 = has_work ? range_begin(w, a.T, a.P) : 0;
    const long long t1 = has_work ? range_begin(w + 1, a.T, a.P) : 0;

    // 1. start the weight stream before anything else
    if (has_work) {
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < S; ++s) mbar_init(&bars[s], 33);   // lane 0's expect_tx + 32 cp.async arrivals
            fence_barrier_init();
        }
        __syncwarp();
        for (int s = 0; s < S && t0 + s < t1; ++s) issue_tile<FMT>(a, L, t0 + s, ring + s * F::STAGE_BYTES, &bars[s], lane);
    }

    // 2. CTA prologue: codebook, x in lane-chunk order, per-chunk sums of x
    if constexpr (FMT == UQ_NF4) {
        if (threadIdx.x < 16) lut[threadIdx.x] = reinterpret_cast<const float*>(a.zc)[threadIdx.x];
    }
    if constexpr (F::NEEDS_SX || XS) {
        const int KBt = L.KB;
        const bool split = (FMT == UQ_INT2_ASYM) && (a.group == 32);
        for (int e = threadIdx.x; e < KBt * M * 32; e += blockDim.x) {
            const int kb = e / (M * 32), m = (e / 32) % M, l = e % 32;
            const int k0 = kb * KT + l * CPL;
            float s0 = 0.f, s1 = 0.f;
            const bool in = k0 < a.K;
            const uint16_t* xp = a.x + (long long)m * a.ldx + k0;
#pragma unroll
            for (int v = 0; v < CPL / 8; ++v) {
                const uint4 q = in ? ldg_nc_v4(xp + 8 * v) : make_uint4(0, 0, 0, 0);
                if constexpr (XS) x_tab[((kb * M + m) * (CPL / 8) + v) * 32 + l] = q;
                if constexpr (F::NEEDS_SX) {
                    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float t = bf16lo_f32(u[j]) + bf16hi_f32(u[j]);
                        if (4 * v + j < CPL / 4) s0 += t; else s1 += t;
                    }
                }
            }
            if constexpr (F::NEEDS_SX) {
                float* row = sx_tab + (long long)kb * F::HALVES * M * 32;
                if (split) {
                    row[m * 32 + l] = s0;
                    row[(M + m) * 32 + l] = s1;
                } else {
                    row[m * 32 + l] = s0 + s1;
                }
            }
        }
    }
    __syncthreads();
    if (!has_work) return;

    const int first_nb = (int)(t0 / L.KB);
    const bool two_groups = (FMT == UQ_INT2_ASYM) && (a.group == 32);
    float acc[RB][M];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

    for (long long t = t0; t < t1; ++t) {
        const int it = (int)(t - t0);
        const int s = it % S;
        const uint32_t parity = (uint32_t)((it / S) & 1);
        const int nb = (int)(t / L.KB), kb = (int)(t % L.KB);
        const int rows = L.rows(nb);
        const int n0 = nb * RB;
        const bool active = lane * CPL < L.width(kb);
        const int k0 = kb * KT + lane * CPL;
        uint8_t* st = ring + s * F::STAGE_BYTES;

        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars[s], parity, a.fault, FAULT_GEMV_WAIT))) {
            // give the copies still in flight a bounded chance to land, then leave
            for (int j = 1; j < S && t + j < t1; ++j) {
                const int sj = (it + j) % S;
                mbar_wait_bounded(&bars[sj], (uint32_t)(((it + j) / S) & 1), a.fault, FAULT_GEMV_WAIT);
            }
            return;
        }
        if (active) {
            RowMeta meta[RB];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                meta[r] = RowMeta{0.f, 0.f, 0.f, 0.f};
                if (r < rows) meta[r] = stage_meta<FMT>(a, L, st, r, n0 + r, kb, lane);
            }
            tile_all_passes<FMT, M, 0, XS>(st, L.slice_bytes(kb), rows, lane, a.x + k0, a.ldx,
                                           x_tab + (long long)kb * M * (CPL / 8) * 32, meta, acc, lut, two_groups,
                                           sx_tab + (long long)kb * F::HALVES * M * 32);
        }
        __syncwarp();
        if (t + S < t1) issue_tile<FMT>(a, L, t + S, st, &bars[s], lane);

        if (kb == L.KB - 1 || t == t1 - 1) {
            // row block done (for this worker): reduce over lanes, then write y or a partial
            const bool full = (kb == L.KB - 1) && (nb != first_nb || (t0 % L.KB) == 0);
            // values padded to a power of two (8 rows x M, M <= 8)
            constexpr int CNT = RB * (M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8);
            float v[CNT];
#pragma unroll
            for (int i = 0; i < CNT; ++i) v[i] = 0.f;
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int m = 0; m < M; ++m) v[r * (CNT / RB) + m] = acc[r][m];
            int idx = 0;
            warp_reduce_transposed<CNT>(v, lane, idx);
            // lane holds the totals of indices idx .. idx + RES - 1; with CNT < 32 several lanes
            // hold the same total and only the first of them writes it
            constexpr int RES = CNT >= 32 ? CNT / 32 : 1;
            constexpr int OWN = CNT >= 32 ? 1 : 32 / CNT;
            const bool owner = (lane % OWN) == 0;
            if (full) {
#pragma unroll
                for (int j = 0; j < RES; ++j) {
                    const int vr = (idx + j) / (CNT / RB), vm = (idx + j) % (CNT / RB);
                    if (owner && vr < rows && vm < M)
                        a.y[(long long)vm * a.ldy + n0 + vr] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
                }
            } else {
                const int slot = 2 * w + (nb == first_nb ? 0 : 1);
                float* part = a.partials + (long long)slot * RB * M;
#pragma unroll
                for (int j = 0; j < RES; ++j) {
                    const int vr = (idx + j) / (CNT / RB), vm = (idx + j) % (CNT / RB);
                    if (owner && vr < rows && vm < M) part[vr * M + vm] = v[j];
                }
                __threadfence();
                __syncwarp();
                unsigned int old = 0;
                if (lane == 0) old = atomicAdd(a.tickets + nb, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                const long long tf = (long long)nb * L.KB;
                const int wf = worker_of(tf, a.T, a.P), wl = worker_of(tf + L.KB - 1, a.T, a.P);
                if (old == (unsigned int)(wl - wf)) {
                    __threadfence();
                    for (int e = lane; e < rows * M; e += 32) {
                        float sum = 0.f;
                        for (int w2 = wf; w2 <= wl; ++w2) {
                            const int nb2 = (int)(range_begin(w2, a.T, a.P) / L.KB);
                            const int slot2 = 2 * w2 + (nb == nb2 ? 0 : 1);
                            sum += __ldcg(a.partials + (long long)slot2 * RB * M + e);
                        }
                        const int r = e / M, m = e % M;
                        a.y[(long long)m * a.ldy + n0 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
                    }
                    if (lane == 0) a.tickets[nb] = 0u;
                }
            }
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int m = 0; m < M; ++m) acc[r][m] = 0.f;
        }
    }
}

inline bool gemv_x_in_smem(int fmt, int K, int M) {
    return gemv_smem_plan(fmt, K, M, true).total <= 227 * 1024;
}
inline size_t gemv_smem_bytes_impl(int fmt, int K, int M) {
    return gemv_smem_plan(fmt, K, M, gemv_x_in_smem(fmt, K, M)).total;
}
inline size_t gemv_partials_floats_impl(int P, int M) { return (size_t)2 * P * RB * M; }

namespace gemv_detail {
template <int FMT, int M, bool XS>
cudaError_t launch_one(const GemvArgs& a, int grid, cudaStream_t st) {
    static bool configured[64] = {};   // the shared-memory opt-in, once per device
    const size_t smem = gemv_smem_plan(FMT, a.K, M, XS).total;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gemv_kernel<FMT, M, XS>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    gemv_kernel<FMT, M, XS><<<grid, GEMV_WARPS * 32, smem, st>>>(a);
    return cudaGetLastError();
}
template <int FMT, int M>
cudaError_t launch_xs(const GemvArgs& a, int grid, cudaStream_t st) {
    if (gemv_x_in_smem(FMT, a.K, M)) return launch_one<FMT, M, true>(a, grid, st);
    return launch_one<FMT, M, false>(a, grid, st);
}
}  // namespace gemv_detail

template <int FMT>
cudaError_t launch_gemv_fmt(const GemvArgs& a, int grid, cudaStream_t st) {
    switch (a.M) {
        case 1: return gemv_detail::launch_xs<FMT, 1>(a, grid, st);
        case 2: return gemv_detail::launch_xs<FMT, 2>(a, grid, st);
        case 3: return gemv_detail::launch_xs<FMT, 3>(a, grid, st);
        case 4: return gemv_detail::launch_xs<FMT, 4>(a, grid, st);
        case 5: return gemv_detail::launch_xs<FMT, 5>(a, grid, st);
        case 6: return gemv_detail::launch_xs<FMT, 6>(a, grid, st);
        case 7: return gemv_detail::launch_xs<FMT, 7>(a, grid, st);
        case 8: return gemv_detail::launch_xs<FMT, 8>(a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace uq
