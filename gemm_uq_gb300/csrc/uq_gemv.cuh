// uq_gemv.cuh -- small-M (M <= 8) fused dequantize + GEMV/GEMM, sm_103a.
//
// "Ultra LLM Engine", section "Fused Kernels": dequantized-weight GEMV for single-token
// decode and GEMM for batched decode.  Decode is bound by streaming the packed weights from
// HBM once; on this GPU the arithmetic of a CUDA-core dot product (unpack, widen, FMA: about
// three issue slots per 4-bit weight) cannot keep up with HBM, so the 4-bit and 2-bit formats
// run on warp-level tensor instructions:
//
//  * gemv_mma_kernel (INT4_SYM, INT4_ASYM, INT2_ASYM, K4).  Work is the list of tiles (16 rows x
//    8 KB of codes), taken in k-major order so a warp's consecutive tiles share their k tile.
//    Either every CTA owns whole 16-row blocks and its warps split their tiles evenly (partial
//    sums of each tile in shared memory, summed per row in k order after one CTA barrier: no
//    second launch), or every warp owns an equal contiguous range of all tiles (stream-K) and
//    stores each tile's partial sums in global memory for gemv_split_reduce, a second launch
//    that sums each row over its k tiles in k order.  Both orders are fixed, so results are
//    bit-reproducible, and no warp ever waits for another.
//  * Each warp keeps a ring of two stages; a stage is one tile's codes plus the tile rows'
//    scales / zero points / K4 records, copied by all 32 lanes with 16-byte (codes: 512
//    contiguous bytes per warp instruction) or 4-byte cp.async in one cp.async group per tile
//    that the warp waits for itself.  With launch overlap the first tile is requested before
//    the wait for the previous kernel on the stream (the weights are constant).
//  * x: one or two rows are copied per warp a k tile at a time (one bulk copy per row, double
//    buffered); more rows are copied whole into shared memory once per CTA, or read through L1
//    when they do not fit.  The sums of x over each scaling group of a k tile are formed once
//    per run of tiles at that k tile.
//  * The packed plane is in mma.m16n8k16 A-fragment order: one 16-byte shared-memory load per
//    lane, a shift and a lop3 per register (magic exponent: bf16 0x4300 | code = 128 + code)
//    give the A fragments, and mma.sync (bf16 x bf16 -> fp32) does the multiply-accumulate and
//    the reduction over the 16-wide k block in one instruction; the M <= 8 activation rows are
//    the instruction's N = 8, so every M <= 8 costs the same.  Per scaling group the fp32 group
//    sum is folded into the row's accumulator:  y += s * (sum x*(128 + q) - (128 + z) * sum x).
//  * gemv_kernel (INT8_SYM, NF4, whose codes do not map onto bf16 exactly by a bit trick): the
//    same layout on CUDA-core FMAs, four stages per warp on mbarriers; the four lanes sharing a
//    row are reduced with warp shuffles, and a row block split between workers is finished by
//    the last contributor (fence + ticket), summing the partials in worker order.
#pragma once
#include "uq_kernels.h"

namespace uq {

template <int FMT> struct GemvFmt {
    static constexpr int BITS = fmt_bits(FMT);
    static constexpr int KT = fmt_kt(FMT);
    static constexpr int KC = fmt_kc(FMT);
    static constexpr int BPC = KC / 16;                            // 16-wide k blocks per chunk
    static constexpr bool MMA = (FMT == UQ_INT4_SYM || FMT == UQ_INT4_ASYM || FMT == UQ_K4 || FMT == UQ_INT2_ASYM);
    static constexpr int GT_MAX = KT / 32;                         // groups per tile row at group 32
    // 32-bit words of metadata staged per tile row: scales (+1 for a misaligned start), zeros
    // (rounded up to 4 words so 16-byte copies land 16-byte aligned)
    static constexpr int SW = (FMT == UQ_K4) ? 16 : (GT_MAX / 2 + 1 + 3) / 4 * 4;
    static constexpr int ZW = (FMT == UQ_INT4_ASYM) ? (GT_MAX / 8 + 1 + 3) / 4 * 4
                            : (FMT == UQ_INT2_ASYM ? (GT_MAX / 2 + 1 + 3) / 4 * 4 : 0);
    static constexpr int MW = SW + ZW;
    static constexpr int META_BYTES = (RB * MW * 4 + 15) / 16 * 16;
    static constexpr int STAGE_BYTES = TILE_BYTES + META_BYTES;
    static constexpr int STAGES = (FMT == UQ_INT2_ASYM) ? 3 : 4;
    static constexpr bool NEEDS_SX = MMA;                          // per-group sums of x
};

// bytes per row of x in shared memory: the row zero-padded to Kp plus 32 bytes, so the rows of a
// B fragment (one 8-byte load per row) fall into different banks
__host__ __device__ inline size_t gemv_x_stride(int Kp) { return (size_t)Kp * 2 + 32; }

// shared-memory plan; identical on host and device
struct GemvSmem {
    size_t bars, lut, sx, ps, x, total;
};
template <int FMT>
__host__ __device__ inline GemvSmem gemv_smem_plan_t(int K, int group, int M, bool x_in_smem) {
    using F = GemvFmt<FMT>;
    const int Kp = (K + F::KC - 1) / F::KC * F::KC;
    const int gs = (FMT == UQ_K4) ? 32 : group;
    GemvSmem p;
    p.bars = (size_t)GEMV_WARPS * F::STAGES * F::STAGE_BYTES;
    p.lut = p.bars + (size_t)(GEMV_WARPS * F::STAGES + 1) * 8;     // + the x mbarrier
    p.sx = p.lut + 64;
    p.x = p.sx + (F::NEEDS_SX ? (size_t)((Kp + gs - 1) / gs) * 8 * 4 : 0);   // sums padded to 8 columns
    p.ps = p.x;
    p.x = (p.x + 127) / 128 * 128;
    p.total = p.x + (x_in_smem ? (size_t)M * gemv_x_stride(Kp) : 0);
    return p;
}
__host__ __device__ inline GemvSmem gemv_smem_plan(int fmt, int K, int group, int M, bool x_in_smem) {
    switch (fmt) {
        case UQ_INT4_SYM: return gemv_smem_plan_t<UQ_INT4_SYM>(K, group, M, x_in_smem);
        case UQ_INT4_ASYM: return gemv_smem_plan_t<UQ_INT4_ASYM>(K, group, M, x_in_smem);
        case UQ_INT8_SYM: return gemv_smem_plan_t<UQ_INT8_SYM>(K, group, M, x_in_smem);
        case UQ_INT2_ASYM: return gemv_smem_plan_t<UQ_INT2_ASYM>(K, group, M, x_in_smem);
        case UQ_NF4: return gemv_smem_plan_t<UQ_NF4>(K, group, M, x_in_smem);
        default: return gemv_smem_plan_t<UQ_K4>(K, group, M, x_in_smem);
    }
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
__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
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
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// D += A * B for one 16 x 8 x 16 block (bf16 inputs, fp32 accumulate)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B (accumulator input zero)
__device__ __forceinline__ void mma_bf16_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    const float z = 0.f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

// Copy the 4-byte-aligned words covering bytes [lo, lo + len) of `base` into dst (word 0 holds
// byte lo & ~3).  A word that would reach past `end` (the array's end) is assembled from plain
// byte loads instead, so nothing outside the caller's buffer is read.
__device__ __forceinline__ void stage_words(uint32_t* dst, const uint8_t* base, long long lo, int len,
                                            long long end, int j) {
    const long long w0 = lo & ~3ll;
    const long long src = w0 + 4ll * j;
    if (len <= 0 || src >= lo + len) return;
    if (src + 4 <= end) {
        cp_async4(dst + j, base + src);
    } else {
        uint32_t v = 0;
        for (int b = 0; b < 4; ++b)
            if (src + b < end) v |= (uint32_t)__ldg(base + src + b) << (8 * b);
        dst[j] = v;
    }
}

// Per-kernel constants of the metadata layout (divisions done once).
struct MetaConst {
    int G;            // scale groups per row (flat formats)
    int GT;           // groups per full tile row
    int ZB;           // bytes of INT4 zero nibbles per row
    int S4;           // K4 super-blocks per row
    bool aligned;     // every tile row's scale slice is 16-byte aligned and a multiple of 16 bytes
};

// One weight's packed codes and metadata (the gated kernel reads two: gate and up).
struct GemvSrc {
    const uint8_t* wq;
    const uint8_t* scales;
    const uint8_t* zc;
};

// Issue the copies of tile t into stage buffer `st` (all lanes take part).  Either the codes come
// as one bulk copy counted on `bar` (transaction bytes) and the metadata copies arrive on `bar`
// too (33 arrivals in all: one per lane when its copies land, and the codes' expect_tx), or, with
// GROUP, everything is 16-byte cp.async (codes: 512 contiguous bytes per warp instruction) in one
// cp.async group per lane that the issuing warp itself waits for (`bar` unused).  The per-lane
// copies keep more of the tile stream in flight than one 8 KB bulk copy per tile: the copy engine
// takes bulk copies one after another, at well under an SM's share of HBM bandwidth at this size.
// GTC: the groups per tile row when the caller knows them at compile time (0: mc.GT at run time).
template <int FMT, bool GROUP = false, int GTC = 0>
__device__ __forceinline__ void issue_tile(const GemvArgs& a, const GemvSrc& w, const Layout& L, const MetaConst& mc, int nb, int kb,
                                           uint8_t* st, uint64_t* bar, int lane) {
    using F = GemvFmt<FMT>;
    const int n0 = nb * RB;
    const int rows = (a.N - n0) < RB ? (a.N - n0) : RB;            // rows with metadata
    uint32_t* md = reinterpret_cast<uint32_t*>(st + TILE_BYTES);
    if constexpr (FMT == UQ_K4) {
        // 16-byte records: one per 256 k of the tile row that lies inside K
        const int sb0 = kb * (F::KT / 256);
        int recs = mc.S4 - sb0;
        if (recs > F::KT / 256) recs = F::KT / 256;
        for (int e = lane; e < rows * recs; e += 32) {
            const int r = e / recs, j = e % recs;
            cp_async16(md + r * F::MW + 4 * j, w.scales + ((long long)(n0 + r) * mc.S4 + sb0 + j) * 16);
        }
    } else if (mc.aligned) {
        // scale slices of GT halves (16-byte multiples, 16-byte aligned): 16-byte copies; INT4
        // zero slices of GT/2 bytes: 4-byte copies; INT2 zero slices like the scales
        const int GT = GTC ? GTC : mc.GT;
        const int sv = GT / 8;                          // 16-byte vectors of scales per row
        const int zv = (FMT == UQ_INT4_ASYM) ? GT / 8 : ((FMT == UQ_INT2_ASYM) ? sv : 0);
        const int per = sv + zv;
        for (int e = lane; e < rows * per; e += 32) {
            const int r = e / per, j = e % per;
            const long long n = n0 + r;
            if (j < sv) {
                cp_async16(md + r * F::MW + 4 * j, w.scales + (n * mc.G + (long long)kb * GT) * 2 + 16 * j);
            } else if constexpr (FMT == UQ_INT4_ASYM) {
                cp_async4(md + r * F::MW + F::SW + (j - sv),
                          w.zc + n * mc.ZB + (long long)kb * (GT >> 1) + 4 * (j - sv));
            } else if constexpr (FMT == UQ_INT2_ASYM) {
                cp_async16(md + r * F::MW + F::SW + 4 * (j - sv), w.zc + (n * mc.G + (long long)kb * GT) * 2 + 16 * (j - sv));
            }
        }
    } else {
        int gc = mc.G - kb * mc.GT;                     // groups of this tile row inside K
        if (gc > mc.GT) gc = mc.GT;
        const long long send = (long long)a.N * mc.G * 2;
        for (int e = lane; e < rows * F::MW; e += 32) {
            const int r = e / F::MW, j = e % F::MW;
            const long long n = n0 + r;
            if (j < F::SW) {
                stage_words(md + r * F::MW, w.scales, (n * mc.G + (long long)kb * mc.GT) * 2, gc * 2, send, j);
            } else if constexpr (FMT == UQ_INT4_ASYM) {
                stage_words(md + r * F::MW + F::SW, w.zc, n * mc.ZB + (long long)kb * (mc.GT >> 1), (gc + 1) >> 1,
                            (long long)a.N * mc.ZB, j - F::SW);
            } else if constexpr (FMT == UQ_INT2_ASYM) {
                stage_words(md + r * F::MW + F::SW, w.zc, (n * mc.G + (long long)kb * mc.GT) * 2, gc * 2, send,
                            j - F::SW);
            }
        }
    }
    if constexpr (GROUP) {
        const int bytes = (int)L.tile_bytes(kb);
        const uint8_t* src = w.wq + L.tile_offset(nb, kb);
        for (int off = lane * 16; off < bytes; off += 512) cp_async16(st + off, src + off);
        cp_async_commit_group();
        (void)bar;
    } else {
        cp_async_arrive_noinc(bar);
        __syncwarp();
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)L.tile_bytes(kb);
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(st, w.wq + L.tile_offset(nb, kb), bytes, bar);
        }
    }
}

// Pointers to row r's staged scales (fp16) and zero points for tile kb: the staged words start
// at the word holding the row's first group, so only the parity / low bits of its offset matter.
template <int FMT>
struct RowPtrs {
    const uint16_t* s;
    const uint8_t* z;
};
template <int FMT>
__device__ __forceinline__ RowPtrs<FMT> row_ptrs(const uint8_t* st, const MetaConst& mc, int r, int n, int kb) {
    using F = GemvFmt<FMT>;
    const uint8_t* row = st + TILE_BYTES + r * F::MW * 4;
    const unsigned first = (unsigned)n * (unsigned)mc.G + (unsigned)kb * (unsigned)mc.GT;   // low bits only
    RowPtrs<FMT> p;
    p.s = reinterpret_cast<const uint16_t*>(row + 2 * (first & 1u));
    if constexpr (FMT == UQ_INT4_ASYM) {
        const unsigned zfirst = (unsigned)n * (unsigned)mc.ZB + (unsigned)kb * (unsigned)(mc.GT >> 1);
        p.z = row + F::SW * 4 + (zfirst & 3u);
    } else if constexpr (FMT == UQ_INT2_ASYM) {
        p.z = row + F::SW * 4 + 2 * (first & 1u);
    } else {
        p.z = row;
    }
    return p;
}

// scale and (128 + z) of a row for the tile's local group li (flat formats)
template <int FMT>
__device__ __forceinline__ void row_meta(const RowPtrs<FMT>& p, int li, float& s, float& zc) {
    s = half_bits_f32(p.s[li]);
    if constexpr (FMT == UQ_INT4_SYM) {
        zc = 136.0f;
    } else if constexpr (FMT == UQ_INT4_ASYM) {
        const uint32_t b = p.z[li >> 1];
        // fp32 with exponent 134 and z at mantissa bits 16..19 is exactly 128 + z
        zc = __uint_as_float(0x43000000u | (((li & 1) ? (b >> 4) : (b & 15u)) << 16));
    } else if constexpr (FMT == UQ_INT2_ASYM) {
        zc = 128.0f + half_bits_f32(reinterpret_cast<const uint16_t*>(p.z)[li]);
    } else {
        zc = 0.0f;
    }
}

// K4: d*sc and dmin*m of row r for the tile's local 32-k sub-block li
__device__ __forceinline__ void row_meta_k4(const uint8_t* st, int r, int li, float& dsc, float& dmm) {
    const uint8_t* row = st + TILE_BYTES + r * GemvFmt<UQ_K4>::MW * 4;
    const uint4 rec = *reinterpret_cast<const uint4*>(row + 16 * (li >> 3));
    const int j = li & 7;
    const uint64_t sc48 = (uint64_t)rec.y | ((uint64_t)(rec.z & 0xFFFFu) << 32);
    const uint64_t m48 = (uint64_t)(rec.z >> 16) | ((uint64_t)rec.w << 16);
    dsc = half_bits_f32((uint16_t)(rec.x & 0xFFFF)) * (float)((sc48 >> (6 * j)) & 63);
    dmm = half_bits_f32((uint16_t)(rec.x >> 16)) * (float)((m48 >> (6 * j)) & 63);
}

}  // namespace

template <int FMT, int M, bool XS>
__global__ void __launch_bounds__(GEMV_WARPS * 32, 1) gemv_kernel(const GemvArgs a) {
    using F = GemvFmt<FMT>;
    constexpr int KT = F::KT, S = F::STAGES, BPC = F::BPC;
    extern __shared__ __align__(128) uint8_t smem[];
    const GemvSmem plan = gemv_smem_plan_t<FMT>(a.K, a.group, M, XS);
    uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + plan.bars);
    float* lut = reinterpret_cast<float*>(smem + plan.lut);
    float* sxg = reinterpret_cast<float*>(smem + plan.sx);
    uint8_t* xs = smem + plan.x;                                   // x rows (+ a zero row), stride xstride
    uint64_t* xbar = bars_all + GEMV_WARPS * S;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int w = blockIdx.x * GEMV_WARPS + warp;
    const bool has_work = w < a.P;
    const Layout L(a.N, a.K, FMT);
    const int gs = (FMT == UQ_K4) ? 32 : a.group;                 // scaling granularity along k
    MetaConst mc;
    mc.G = a.K / a.group;
    mc.GT = KT / a.group;
    mc.ZB = (mc.G + 1) >> 1;
    mc.S4 = a.K / 256;
    const int bpg = gs / 16;                                       // 16-k blocks per group: 2, 4 or 8
    const int bpg_log = bpg == 2 ? 1 : (bpg == 4 ? 2 : 3);
    const size_t xstride = gemv_x_stride(L.Kp);
    // 16-byte metadata copies: row slices 16-byte aligned and a multiple of 16 bytes long
    mc.aligned = (a.K % (8 * a.group)) == 0 && (mc.GT % 8) == 0;
    uint8_t* ring = smem + (size_t)warp * S * F::STAGE_BYTES;
    uint64_t* bars = bars_all + warp * S;
    const long long t0 = has_work ? range_begin(w, a.T, a.P) : 0;
    const long long t1 = has_work ? range_begin(w + 1, a.T, a.P) : 0;

    // 0. let the next kernel on the stream start launching (it only prefetches its own weights
    //    before it waits for this grid; no effect unless launched with launch overlap)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // 1. start the weight stream before anything else (weights and metadata are constant)
    if (has_work) {
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < S; ++s) mbar_init(&bars[s], 33);   // lane 0's expect_tx + 32 cp.async arrivals
            fence_barrier_init();
        }
        __syncwarp();
        int inb = (int)(t0 / L.KB), ikb = (int)(t0 % L.KB);
        for (int s = 0; s < S && t0 + s < t1; ++s) {
            issue_tile<FMT>(a, GemvSrc{a.wq, a.scales, a.zc}, L, mc, inb, ikb, ring + s * F::STAGE_BYTES, &bars[s], lane);
            if (++ikb == L.KB) { ikb = 0; ++inb; }
        }
    }

    // 2. everything below may depend on the previous kernel on the stream (x, the split-K
    //    workspace, y): wait for it to complete (returns at once when not launched overlapped)
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // CTA prologue: codebook, x rows, per-group sums of x
    if constexpr (FMT == UQ_NF4) {
        if (threadIdx.x < 16) lut[threadIdx.x] = reinterpret_cast<const float*>(a.zc)[threadIdx.x];
    }
    if constexpr (XS) {
        // one bulk copy per row of x into shared memory (rows are K * 2 bytes, a multiple of 16);
        // the pad [K, Kp) of every row is zero
        if (threadIdx.x == 0) {
            mbar_init(xbar, 1);
            fence_barrier_init();
            mbar_arrive_expect_tx(xbar, (uint32_t)(M * a.K * 2));
#pragma unroll
            for (int m = 0; m < M; ++m) bulk_g2s(xs + m * xstride, a.x + (long long)m * a.ldx, (uint32_t)(a.K * 2), xbar);
        }
        const int padw = (L.Kp - a.K) / 2;                          // 32-bit words of pad per row
        for (int e = threadIdx.x; e < M * padw; e += blockDim.x)
            reinterpret_cast<uint32_t*>(xs + (e / padw) * xstride + a.K * 2)[e % padw] = 0u;
        __syncthreads();
        // on a timeout the fault word is set and the kernel goes on (its results are then
        // meaningless) so the ring's copies in flight are still drained below
        mbar_wait_bounded(xbar, 0, a.fault, FAULT_GEMV_WAIT);
    }
    if constexpr (F::NEEDS_SX) {
        // sxg[gi * 8 + m] = sum of x[m][k] over group gi (k < K), in k order; 0 for m >= M
        const int gp = (L.Kp + gs - 1) / gs;
        for (int e = threadIdx.x; e < gp * 8; e += blockDim.x) {
            const int gi = e >> 3, m = e & 7;
            float s0 = 0.f;
            if (m < M) {
                const int kend = (gi * gs + gs) < a.K ? (gi * gs + gs) : a.K;
                for (int k = gi * gs; k < kend; k += 8) {
                    uint4 q;
                    if constexpr (XS) q = *reinterpret_cast<const uint4*>(xs + m * xstride + k * 2);
                    else q = ldg_nc_v4(a.x + (long long)m * a.ldx + k);
                    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) s0 += bf16lo_f32(u[j]) + bf16hi_f32(u[j]);
                }
            }
            sxg[e] = s0;
        }
    }
    __syncthreads();
    if (!has_work) return;

    const int first_nb = (int)(t0 / L.KB);
    // MMA path: acc[j*2 + e] = row g + 8j, column 2c + e.  FFMA path: accf[j][m] = row g + 8j.
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float accf[2][M];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int m = 0; m < M; ++m) accf[j][m] = 0.f;

    // (row block, k tile) of the tile being consumed and of the next one to prefetch, advanced
    // incrementally (no 64-bit division per tile)
    int nb = (int)(t0 / L.KB), kb = (int)(t0 % L.KB);
    int pnb = nb, pkb = kb;
    for (int s = 0; s < S; ++s)
        if (++pkb == L.KB) { pkb = 0; ++pnb; }
    for (long long t = t0; t < t1; ++t) {
        const int it = (int)(t - t0);
        const int s = it % S;
        const uint32_t parity = (uint32_t)((it / S) & 1);
        const int n0 = nb * RB;
        uint8_t* st = ring + s * F::STAGE_BYTES;
        const int nchunks = L.chunks(kb);
        const int blk0 = (kb * KT) / 16;                           // first global 16-k block of the tile

        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars[s], parity, a.fault, FAULT_GEMV_WAIT))) {
            // give the copies still in flight a bounded chance to land, then leave
            for (int j = 1; j < S && t + j < t1; ++j) {
                const int sj = (it + j) % S;
                mbar_wait_bounded(&bars[sj], (uint32_t)(((it + j) / S) & 1), a.fault, FAULT_GEMV_WAIT);
            }
            return;
        }

        static_assert(!F::MMA, "the 4-bit and 2-bit formats run gemv_mma_kernel");
        {
            // CUDA-core path (INT8_SYM, NF4): lane holds rows g and g + 8 at k = 16 blk + 4c .. +3
            const int G_all = mc.G;
            RowPtrs<FMT> rp[2];
            rp[0] = row_ptrs<FMT>(st, mc, g, n0 + g, kb);
            rp[1] = row_ptrs<FMT>(st, mc, g + 8, n0 + g + 8, kb);
            float p[2][M];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m) p[j][m] = 0.f;
            for (int q = 0; q < nchunks; ++q) {
                const uint4 cw = *reinterpret_cast<const uint4*>(st + q * CHUNK + lane * 16);
                const uint32_t wv[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int bi = 0; bi < BPC; ++bi) {
                    const int lb = q * BPC + bi;
                    const int blk = blk0 + lb;
                    float cv[2][4];
                    if constexpr (FMT == UQ_INT8_SYM) {
#pragma unroll
                        for (int j = 0; j < 2; ++j)
#pragma unroll
                            for (int e = 0; e < 4; ++e) cv[j][e] = byte_magic_f32(wv[2 * bi + j], e) - 8388736.0f;
                    } else {
                        const uint32_t wd = wv[bi];
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp) {
                            // pair pp: row g + 8 (pp & 1), k = 4c + 2 (pp >> 1) + {0, 1}
                            cv[pp & 1][2 * (pp >> 1)] = lut[(wd >> (4 * pp)) & 15u];
                            cv[pp & 1][2 * (pp >> 1) + 1] = lut[(wd >> (16 + 4 * pp)) & 15u];
                        }
                    }
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        uint2 xb;
                        xb = make_uint2(0, 0);
                        if (blk * 16 + 4 * c < a.K) {
                            if constexpr (XS) xb = *reinterpret_cast<const uint2*>(xs + m * xstride + (blk * 16 + 4 * c) * 2);
                            else xb = ldg_nc_v2(a.x + (long long)m * a.ldx + blk * 16 + 4 * c);
                        }
                        const float x0 = bf16lo_f32(xb.x), x1 = bf16hi_f32(xb.x);
                        const float x2 = bf16lo_f32(xb.y), x3 = bf16hi_f32(xb.y);
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            p[j][m] = fmaf(x0, cv[j][0], p[j][m]);
                            p[j][m] = fmaf(x1, cv[j][1], p[j][m]);
                            p[j][m] = fmaf(x2, cv[j][2], p[j][m]);
                            p[j][m] = fmaf(x3, cv[j][3], p[j][m]);
                        }
                    }
                    if (((lb + 1) & (bpg - 1)) == 0) {
                        const int li = lb >> bpg_log;
                        if (kb * mc.GT + li < G_all) {
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                float sc, zc;
                                row_meta<FMT>(rp[j], li, sc, zc);
#pragma unroll
                                for (int m = 0; m < M; ++m) accf[j][m] = fmaf(sc, p[j][m], accf[j][m]);
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 2; ++j)
#pragma unroll
                            for (int m = 0; m < M; ++m) p[j][m] = 0.f;
                    }
                }
            }
        }
        __syncwarp();
        if (t + S < t1) {
            issue_tile<FMT>(a, GemvSrc{a.wq, a.scales, a.zc}, L, mc, pnb, pkb, st, &bars[s], lane);
            if (++pkb == L.KB) { pkb = 0; ++pnb; }
        }

        if (kb == L.KB - 1 || t == t1 - 1) {
            // row block done (for this worker): write y or a partial
            const bool full = (kb == L.KB - 1) && (nb != first_nb || (t0 % L.KB) == 0);
            // this thread's results: rows g + 8j, columns 2c + e (MMA) or all columns (FFMA, lane c == 0)
            float out[2][M];
            bool mine[2][M];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m) { out[j][m] = 0.f; mine[j][m] = false; }
            if constexpr (F::MMA) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
#pragma unroll
                        for (int m = 0; m < M; ++m)
                            if (m == 2 * c + e) { out[j][m] = acc[2 * j + e]; mine[j][m] = true; }
            } else {
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        float v = accf[j][m];
                        v += __shfl_xor_sync(0xffffffffu, v, 1);
                        v += __shfl_xor_sync(0xffffffffu, v, 2);
                        out[j][m] = v;
                        mine[j][m] = (c == 0);
                    }
            }
            if (full) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const int n = n0 + g + 8 * j;
                        if (mine[j][m] && n < a.N)
                            store_out(a, m, n, out[j][m]);
                    }
            } else {
                const int slot = 2 * w + (nb == first_nb ? 0 : 1);
                float* part = a.partials + (long long)slot * RB * M;
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int m = 0; m < M; ++m)
                        if (mine[j][m]) part[(g + 8 * j) * M + m] = out[j][m];
                __threadfence();
                __syncwarp();
                unsigned int old = 0;
                if (lane == 0) old = atomicAdd(a.tickets + nb, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                const long long tf = (long long)nb * L.KB;
                const int wf = worker_of(tf, a.T, a.P), wl = worker_of(tf + L.KB - 1, a.T, a.P);
                if (old == (unsigned int)(wl - wf)) {
                    __threadfence();
                    for (int e = lane; e < RB * M; e += 32) {
                        const int r = e / M, m = e % M;
                        if (n0 + r >= a.N) continue;
                        float sum = 0.f;
                        for (int w2 = wf; w2 <= wl; ++w2) {
                            const int nb2 = (int)(range_begin(w2, a.T, a.P) / L.KB);
                            const int slot2 = 2 * w2 + (nb == nb2 ? 0 : 1);
                            sum += __ldcg(a.partials + (long long)slot2 * RB * M + e);
                        }
                        store_out(a, m, n0 + r, sum);
                    }
                    if (lane == 0) a.tickets[nb] = 0u;
                }
            }
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m) accf[j][m] = 0.f;
        }
        if (++kb == L.KB) { kb = 0; ++nb; }
    }
}


// ------------------------------------------------------------------------------------------------
// 4-bit and 2-bit formats: the GEMV on mma.sync.  GB = 16-k blocks per scaling group (2, 4 or 8;
// K4 uses its 32-weight sub-blocks, GB = 2).  M (1..8) is a runtime value: the instruction always
// computes 8 columns, so the work per weight does not depend on it.
//
// Per 16 x 16 block of weights a lane issues its share of a 16-byte code load, four lop3 (three
// after a shift) to form the A fragment, one 8-byte load of x and the mma.  Per group: two fp32
// FMAs per accumulator with the group's scale and zero-point term, the latter using the group's
// sum of x.
//
// Tile order is k-major: tile i of a range is (k tile i / R, row block i % R) for R row blocks, so
// a warp's consecutive tiles share their k tile.  The sums of x over the k tile's groups (an mma
// chain with A = 1) are computed once per run of equal k tile instead of once per tile, and with
// one or two rows of x the warp copies only that k tile's slice of x, once per run.  Every tile's
// partial sums are stored (shared memory when the CTA owns whole row blocks, global memory
// otherwise) and summed over the k tiles in a fixed order afterwards.
// Two CTAs of 4 warps per SM (INT2: 3) rather than one of 8: the same warps per SM, and each
// CTA's shared memory (~105 KB) leaves room for a CTA of the next kernel on the stream, which with
// launch overlap starts streaming its weights while this kernel's last CTAs finish.
template <int FMT> struct MmaCfg {
    static constexpr int WARPS = (FMT == UQ_INT2_ASYM) ? 3 : 4;    // workers per CTA
    static constexpr int STAGES = 2;                               // tiles in flight per worker
};
constexpr int MMA_CTAS_PER_SM = 2;
constexpr int MMA_TPW = 6;        // tiles per warp at most when the CTA owns whole row blocks

// bytes per row of x in shared memory: 32 bytes of padding put the four rows a half-warp's 8-byte
// B-fragment loads touch into different banks
__host__ __device__ inline size_t gemv_mma_x_stride(int Kp) { return (size_t)Kp * 2 + 32; }

// Where the mma GEMV reads x (template parameter XM):
//   MMA_X_GLOBAL  straight from global memory (through L1);
//   MMA_X_WHOLE   all of x copied into shared memory once per CTA, before the first tile;
//   MMA_X_SLICE   each warp copies the slice of x of its current k tile (KT k of every row) into a
//                 buffer of its own, the next run's slice while the current run computes.
constexpr int MMA_X_GLOBAL = 0, MMA_X_WHOLE = 1, MMA_X_SLICE = 2;
// bytes per row of an x slice (row padding as for the whole x when there are several rows)
__host__ __device__ inline int gemv_mma_xslice_stride(int fmt, int M) {
    return M <= 1 ? fmt_kt(fmt) * 2 : fmt_kt(fmt) * 2 + 32;
}

// Shared memory: rings [warps][stages][stage] | ring and x mbarriers | sums of x [warps][groups of
// a tile][8] | partial sums [tiles of the CTA, at most warps x MMA_TPW][16][8] | x (whole, or
// [warps][2][M] slices)
__host__ __device__ inline GemvSmem gemv_mma_smem_plan(int fmt, int K, int group, int M, int xm) {
    int stage = 0, warps = 0;
    const int kc = fmt_kc(fmt), kt = fmt_kt(fmt);
    switch (fmt) {
        case UQ_INT4_SYM: stage = GemvFmt<UQ_INT4_SYM>::STAGE_BYTES; warps = MmaCfg<UQ_INT4_SYM>::WARPS; break;
        case UQ_INT4_ASYM: stage = GemvFmt<UQ_INT4_ASYM>::STAGE_BYTES; warps = MmaCfg<UQ_INT4_ASYM>::WARPS; break;
        case UQ_INT2_ASYM: stage = GemvFmt<UQ_INT2_ASYM>::STAGE_BYTES; warps = MmaCfg<UQ_INT2_ASYM>::WARPS; break;
        default: stage = GemvFmt<UQ_K4>::STAGE_BYTES; warps = MmaCfg<UQ_K4>::WARPS; break;
    }
    const int stages = 2;
    const int Kp = (K + kc - 1) / kc * kc;
    const int gs = (fmt == UQ_K4) ? 32 : group;
    GemvSmem p;
    p.bars = (size_t)warps * stages * stage;
    p.lut = p.bars + (size_t)(warps * stages + 2 * warps + 1) * 8;  // ring, x-slice and whole-x mbarriers
    p.sx = (p.lut + 15) / 16 * 16;
    p.ps = p.sx + (size_t)warps * (kt / gs) * 8 * 4;
    p.x = (p.ps + (size_t)warps * MMA_TPW * RB * 8 * 4 + 127) / 128 * 128;
    p.total = p.x;
    if (xm == MMA_X_WHOLE) p.total += (size_t)M * gemv_mma_x_stride(Kp);
    if (xm == MMA_X_SLICE) p.total += (size_t)warps * 2 * M * gemv_mma_xslice_stride(fmt, M);
    return p;
}
// x slices for one or two rows, else the whole x if it fits, else global memory (each within the
// shared memory that keeps MMA_CTAS_PER_SM CTAs on an SM)
constexpr int MMA_SMEM_LIMIT = (228 * 1024) / MMA_CTAS_PER_SM - 1024;
__host__ __device__ inline int gemv_mma_xmode(int fmt, int K, int group, int M) {
    if (M <= 2 && gemv_mma_smem_plan(fmt, K, group, M, MMA_X_SLICE).total <= MMA_SMEM_LIMIT) return MMA_X_SLICE;
    if (gemv_mma_smem_plan(fmt, K, group, M, MMA_X_WHOLE).total <= MMA_SMEM_LIMIT) return MMA_X_WHOLE;
    return MMA_X_GLOBAL;
}

// GATED: the gated projection in one launch.  The work list interleaves the gate and up weights' row
// blocks (work row block 2j = gate row block j, 2j + 1 = up row block j), every CTA owns whole pairs,
// and the per-row reduction forms h = silu(g) * u (or the second pass does, for the stream-K split).
template <int FMT, int GB, int XM, bool GATED>
__global__ void __launch_bounds__(MmaCfg<FMT>::WARPS * 32, MMA_CTAS_PER_SM) gemv_mma_kernel(const GemvArgs a) {
    using F = GemvFmt<FMT>;
    constexpr int KT = F::KT, S = MmaCfg<FMT>::STAGES, W = MmaCfg<FMT>::WARPS;
    constexpr int GS = GB * 16;                                     // k per scaling group
    constexpr int GPT = KT / GS;                                    // groups per full tile row
    constexpr int WPG = (FMT == UQ_INT2_ASYM) ? GB / 2 : GB;        // code words per lane per group
    constexpr int BPCH = F::BPC;                                    // 16-k blocks per 512-byte chunk
    constexpr bool XS = XM == MMA_X_WHOLE;
    constexpr uint32_t ONES = 0x3F803F80u;                          // bf16 pair (1, 1)
    extern __shared__ __align__(128) uint8_t smem[];
    const int M = a.M;
    const GemvSmem plan = gemv_mma_smem_plan(FMT, a.K, a.group, M, XM);
    const int XB = gemv_mma_xslice_stride(FMT, M);                 // x slice: bytes per row
    uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + plan.bars);
    uint8_t* xs = smem + plan.x;
    float* cpart = reinterpret_cast<float*>(smem + plan.ps);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const Layout L(a.N, a.K, FMT);
    uint8_t* ring = smem + (size_t)warp * S * F::STAGE_BYTES;
    uint64_t* bars = bars_all + warp * S;
    uint64_t* xsl_bar = bars_all + W * S + 2 * warp;               // this warp's two x-slice buffers
    uint64_t* xbar = bars_all + W * S + 2 * W;                      // the whole x
    float* sxw = reinterpret_cast<float*>(smem + plan.sx) + warp * GPT * 8;   // sums of x of the run's k tile
    uint8_t* xsl = xs + (size_t)warp * 2 * M * XB;                  // this warp's x-slice buffers

    // Work split.  cta_rows: CTA b owns row blocks [rb0, rb1), R of them, and its W warps split the
    // R * KB tiles evenly; otherwise worker w = CTA + grid * warp (strided, so a small matrix still
    // spreads over every SM) owns an equal share of all NB * KB tiles.  Tile i -> (k tile i / R,
    // row block i % R) with R = NB for the whole matrix.
    constexpr int WU = GATED ? 2 : 1;                              // work row blocks per weight row block
    const bool cta_rows = a.cta_rows != 0;
    const int NBU = a.NB / WU;                                      // pairs (gated) or row blocks
    const int rb0 = cta_rows ? WU * (int)((long long)blockIdx.x * NBU / gridDim.x) : 0;
    const int R = cta_rows ? WU * (int)((long long)(blockIdx.x + 1) * NBU / gridDim.x) - rb0 : a.NB;
    const unsigned Tc = (unsigned)(R * L.KB);                       // the CTA's tiles (cta_rows; small)
    const int w = cta_rows ? warp : (int)(blockIdx.x + gridDim.x * warp);
    const bool has_work = cta_rows ? true : w < a.P;
    const long long t0 = cta_rows ? (long long)(warp * Tc / W) : (has_work ? range_begin(w, a.T, a.P) : 0);
    const long long t1 = cta_rows ? (long long)((warp + 1) * Tc / W) : (has_work ? range_begin(w + 1, a.T, a.P) : 0);
    int ntl = (int)(t1 - t0);                                       // this warp's tiles
    if (cta_rows && ntl > MMA_TPW) {                                // the host never splits this way
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
    const int G_all = a.K / GS;                                     // real scaling groups per row
    const size_t xstride = gemv_mma_x_stride(L.Kp);
    const int kb_first = ntl > 0 ? kb_of(t0) : 0;
    const int kb_last = ntl > 0 ? kb_of(t1 - 1) : -1;

    // x slice of k tile kb into buffer `slot` (lane 0)
    auto issue_xslice = [&](int kb, int slot) {
        const int kx = (a.K - kb * KT) < KT ? (a.K - kb * KT) : KT;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&xsl_bar[slot], (uint32_t)(M * kx * 2));
        for (int m = 0; m < M; ++m)
            bulk_g2s(xsl + (slot * M + m) * XB, a.x + (long long)m * a.ldx + (long long)kb * KT, (uint32_t)(kx * 2),
                     &xsl_bar[slot]);
    };

    // ---- prologue.  The weights and their metadata are constant: with launch overlap they are
    // requested before the wait for the previous kernel (which may write x); x after it.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (has_work && lane == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        mbar_init(&xsl_bar[0], 1);
        mbar_init(&xsl_bar[1], 1);
        fence_barrier_init();
    }
    if (XS && threadIdx.x == 0) {
        mbar_init(xbar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    int issued = 0;                                                 // tiles requested so far
    // the weight and weight row block of a work row block
    const GemvSrc src_gate{a.wq, a.scales, a.zc}, src_up{a.wq2, a.scales2, a.zc2};
    // k-major tile coordinates (k tile, row block index in [0, R)) are advanced incrementally: a
    // 64-bit division per tile would cost more than the tile's scale folds
    int ikb = ntl > 0 ? kb_of(t0) : 0, irb = ntl > 0 ? (int)(t0 % R) : 0;   // the next tile to request
    auto issue_next = [&]() {
        const int nbw = rb0 + irb;
        issue_tile<FMT, true, GPT>(a, (GATED && (nbw & 1)) ? src_up : src_gate, L, mc, GATED ? nbw >> 1 : nbw, ikb,
                                   ring + (issued % S) * F::STAGE_BYTES, &bars[issued % S], lane);
        if (++irb == R) { irb = 0; ++ikb; }
        ++issued;
    };
    // Only the first tile before the sums of x of the first run: at the start every warp of the
    // GPU requests its tiles at once and a copy's issue waits for room in the memory system, so
    // the second tile is requested once this warp's sums of x are done (the memory system is
    // still busy with the first tiles then).
    if (a.overlap && has_work && ntl > 0) issue_next();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int xissued = 0;                                                // x-slice runs requested so far
    if constexpr (XM == MMA_X_SLICE) {
        if (has_work && ntl > 0 && lane == 0) {
            issue_xslice(kb_first, 0);
            if (kb_last > kb_first) issue_xslice(kb_first + 1, 1);
        }
        xissued = (ntl > 0) ? ((kb_last > kb_first) ? 2 : 1) : 0;
    }
    if constexpr (XS) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(xbar, (uint32_t)(M * a.K * 2));
            for (int m = 0; m < M; ++m) bulk_g2s(xs + m * xstride, a.x + (long long)m * a.ldx, (uint32_t)(a.K * 2), xbar);
        }
        __syncthreads();                            // no warp's weight copies ahead of x
    }
    if (has_work && issued == 0 && ntl > 0) issue_next();
    if constexpr (XS) {
        const int padw = (L.Kp - a.K) / 2;
        for (int e = threadIdx.x; e < M * padw; e += blockDim.x)
            reinterpret_cast<uint32_t*>(xs + (e / padw) * xstride + a.K * 2)[e % padw] = 0u;
        __syncthreads();                            // the zero padding is visible
        mbar_wait_bounded(xbar, 0, a.fault, FAULT_GEMV_WAIT);
    }
    if (!has_work) return;                          // (never in cta_rows mode: every warp meets the end barrier)

    float acc[4] = {0.f, 0.f, 0.f, 0.f};        // rows g + 8j, columns 2c + e
    const int mrow = g < M ? g : M - 1;          // B rows beyond M repeat a real row; their D columns are unused
    const uint16_t* xgrow = a.x + (long long)mrow * a.ldx + 4 * c;
    int cur_kb = -1, run = -1;
    const uint8_t* xt = nullptr;                 // this lane's x at the current k tile's first k
    const uint16_t* xgt = xgrow;

    int ckb = ntl > 0 ? kb_of(t0) : 0, crb = ntl > 0 ? (int)(t0 % R) : 0;   // the tile being consumed
    for (int li = 0; li < ntl; ++li) {
        const long long i = t0 + li;
        const int kb = ckb, nb = GATED ? (rb0 + crb) >> 1 : rb0 + crb;
        if (++crb == R) { crb = 0; ++ckb; }
        const int n0 = nb * RB;
        const int gi0 = kb * GPT;
        const int ng = (G_all - gi0) < GPT ? (G_all - gi0) : GPT;   // groups of the tile inside K
        if (kb != cur_kb) {
            // a new run of tiles at k tile kb: its x, then the sums of x over its groups
            cur_kb = kb;
            ++run;
            if constexpr (XM == MMA_X_SLICE) {
                const int slot = run & 1;
                bool ok = mbar_wait_bounded(&xsl_bar[slot], (uint32_t)((run >> 1) & 1), a.fault, FAULT_GEMV_WAIT);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (run >= 1 && kb + 1 <= kb_last) {
                    __syncwarp();                                   // the buffer's previous run is done
                    if (lane == 0) issue_xslice(kb + 1, slot ^ 1);
                    ++xissued;
                }
                xt = xsl + (slot * M + mrow) * XB + 8 * c;
            } else {
                xt = xs + mrow * xstride + 8 * c + (size_t)kb * KT * 2;
            }
            xgt = xgrow + (long long)kb * KT;
            __syncwarp();                                           // the previous run's sums are read
            if constexpr (XM == MMA_X_SLICE) {
                // one or two rows: lane l adds up k = KL l .. KL l + KL - 1 of each row in fp32 (a
                // group spans GS / KL lanes, combined by shuffles, or a lane spans KL / GS groups)
                constexpr int KL = KT / 32;
                const int slot = run & 1;
                for (int m = 0; m < M; ++m) {
                    const uint4* xp = reinterpret_cast<const uint4*>(xsl + (slot * M + m) * XB + lane * KL * 2);
                    constexpr int NGL = (KL / GS) > 1 ? (KL / GS) : 1;  // groups within the lane's k
                    float gsum[NGL];
#pragma unroll
                    for (int q = 0; q < NGL; ++q) gsum[q] = 0.f;
#pragma unroll
                    for (int v = 0; v < KL / 8; ++v) {
                        const uint4 w4 = xp[v];
                        const uint32_t wv4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const int q = (NGL > 1) ? (v * 8 + 2 * h) / GS : 0;
                            gsum[q] += __uint_as_float(wv4[h] << 16) + __uint_as_float(wv4[h] & 0xFFFF0000u);
                        }
                    }
                    if constexpr (GS >= KL) {
#pragma unroll
                        for (int o = 1; o < GS / KL; o <<= 1) gsum[0] += __shfl_xor_sync(0xffffffffu, gsum[0], o);
                        if ((lane & (GS / KL - 1)) == 0) sxw[(lane / (GS / KL)) * 8 + m] = gsum[0];
                    } else {
#pragma unroll
                        for (int q = 0; q < NGL; ++q) sxw[(lane * NGL + q) * 8 + m] = gsum[q];
                    }
                }
            } else {
            for (int gg = 0; gg < ng; ++gg) {
                float ds[2][4];
#pragma unroll
                for (int j = 0; j < GB; ++j) {
                    uint32_t bx, by;
                    if constexpr (XM != MMA_X_GLOBAL) {
                        const uint2 v = *reinterpret_cast<const uint2*>(xt + (gg * GB + j) * 32);
                        bx = v.x; by = v.y;
                    } else {
                        const int kk = (gg * GB + j) * 16;
                        const uint2 v = (kb * KT + kk + 4 * c < a.K) ? ldg_nc_v2(xgt + kk) : make_uint2(0, 0);
                        bx = v.x; by = v.y;
                    }
                    if (j < 2) mma_bf16_zero(ds[j & 1], ONES, ONES, ONES, ONES, bx, by);
                    else mma_bf16(ds[j & 1], ONES, ONES, ONES, ONES, bx, by);
                }
                if (g == 0) {
                    float2 v;
                    v.x = ds[0][0] + ds[1][0];
                    v.y = ds[0][1] + ds[1][1];
                    *reinterpret_cast<float2*>(sxw + gg * 8 + 2 * c) = v;
                }
            }
            }
            __syncwarp();
        }
        while (issued < ntl && issued < li + S) issue_next();        // top up the ring (into stages consumed)
        const int s = li % S;
        uint8_t* st = ring + s * F::STAGE_BYTES;
        // this tile's copies (one cp.async group) are complete once at most the groups of later
        // tiles are pending
        static_assert(S == 2, "one later group at most");
        if (issued > li + 1) cp_async_wait_group<1>();
        else cp_async_wait_group<0>();
        __syncwarp();
        RowPtrs<FMT> rp[2];
        if constexpr (FMT != UQ_K4) {
            rp[0] = row_ptrs<FMT>(st, mc, g, n0 + g, kb);
            rp[1] = row_ptrs<FMT>(st, mc, g + 8, n0 + g + 8, kb);
        }

        auto group_step = [&](const int gg) {
            // this lane's code words for the group's GB blocks
            uint32_t wv[WPG];
            {
                const int blk = gg * GB;                            // first block of the group in the tile
                const uint8_t* cp = st + (blk / BPCH) * CHUNK + lane * 16 + ((blk % BPCH) * WPG / GB) * 4;
                if constexpr (WPG == 4) {
                    const uint4 v = *reinterpret_cast<const uint4*>(cp);
                    wv[0] = v.x; wv[1] = v.y; wv[2] = v.z; wv[3] = v.w;
                } else if constexpr (WPG == 8) {
                    const uint4 v0 = *reinterpret_cast<const uint4*>(cp);
                    const uint4 v1 = *reinterpret_cast<const uint4*>(cp + CHUNK);
                    wv[0] = v0.x; wv[1] = v0.y; wv[2] = v0.z; wv[3] = v0.w;
                    wv[4] = v1.x; wv[5] = v1.y; wv[6] = v1.z; wv[7] = v1.w;
                } else if constexpr (WPG == 2) {
                    const uint2 v = *reinterpret_cast<const uint2*>(cp);
                    wv[0] = v.x; wv[1] = v.y;
                } else {
                    wv[0] = *reinterpret_cast<const uint32_t*>(cp);
                }
            }
            // B fragments: x at k = 16 blk + 4c .. +3 of row mrow (8 bytes per block)
            uint32_t bx[GB], by[GB];
            if constexpr (XM != MMA_X_GLOBAL) {
#pragma unroll
                for (int j = 0; j < GB; ++j) {
                    const uint2 v = *reinterpret_cast<const uint2*>(xt + (gg * GB + j) * 32);
                    bx[j] = v.x; by[j] = v.y;
                }
            } else {
#pragma unroll
                for (int j = 0; j < GB; ++j) {
                    const int kk = (gg * GB + j) * 16;
                    const uint2 v = (kb * KT + kk + 4 * c < a.K) ? ldg_nc_v2(xgt + kk) : make_uint2(0, 0);
                    bx[j] = v.x; by[j] = v.y;
                }
            }
            // the group's sum of (128 + q) x, in two chains (even / odd blocks)
            float dd[2][4];
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
                if (j < 2) mma_bf16_zero(dd[j & 1], a0, a1, a2, a3, bx[j], by[j]);
                else mma_bf16(dd[j & 1], a0, a1, a2, a3, bx[j], by[j]);
            }
            // fold the group into the row sums, with the run's sums of x over the group
            const float2 sxv = *reinterpret_cast<const float2*>(sxw + gg * 8 + 2 * c);
            float d[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) d[e] = dd[0][e] + dd[1][e];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if constexpr (FMT == UQ_K4) {
                    float dsc, dmm;
                    row_meta_k4(st, g + 8 * j, gg, dsc, dmm);
                    const float off = fmaf(128.0f, dsc, dmm);
                    acc[2 * j] = fmaf(dsc, d[2 * j], fmaf(-off, sxv.x, acc[2 * j]));
                    acc[2 * j + 1] = fmaf(dsc, d[2 * j + 1], fmaf(-off, sxv.y, acc[2 * j + 1]));
                } else {
                    float sc, zc;
                    row_meta<FMT>(rp[j], gg, sc, zc);
                    const float szc = sc * zc;
                    acc[2 * j] = fmaf(sc, d[2 * j], fmaf(-szc, sxv.x, acc[2 * j]));
                    acc[2 * j + 1] = fmaf(sc, d[2 * j + 1], fmaf(-szc, sxv.y, acc[2 * j + 1]));
                }
            }
        };
        if (ng == GPT) {
            // 8 groups per step for 32-k groups: a K4 record (8 sub-blocks) is then read and
            // decoded once per row per step, its 6-bit fields at constant shifts
            constexpr int GUNROLL = (GB == 2) ? 8 : 4;
#pragma unroll GUNROLL
            for (int gg = 0; gg < GPT; ++gg) group_step(gg);
        } else {
#pragma unroll 1
            for (int gg = 0; gg < ng; ++gg) group_step(gg);
        }
        __syncwarp();

        // the tile's partial sums: shared memory (cta_rows) or global memory, summed over k tiles later
        if (cta_rows) {
            float* part = cpart + (i * RB) * 8;                     // slot = the tile's index in the CTA's range
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) part[(g + 8 * j) * 8 + 2 * c + e] = acc[2 * j + e];
        } else {
            float* part = a.partials + i * RB * M;
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    if (2 * c + e < M) part[(g + 8 * j) * M + 2 * c + e] = acc[2 * j + e];
        }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    }
    // a wait that timed out (fault flag set) left copies in flight: let them land before leaving
    cp_async_wait_group<0>();
    if constexpr (XM == MMA_X_SLICE) {
        for (int r = (run > 0 ? run : 0); r < xissued; ++r)
            mbar_wait_bounded(&xsl_bar[r & 1], (uint32_t)((r >> 1) & 1), a.fault, FAULT_GEMV_WAIT);
    }
    if (!cta_rows) return;
    // cta_rows: each row's sum over the k tiles, in k order, from the warps that computed them
    __syncthreads();
    auto row_sum = [&](int rbi, int r, int m) {
        float sum = 0.f;
        for (int kb = 0; kb < L.KB; ++kb) sum += cpart[((kb * R + rbi) * RB + r) * 8 + m];
        return sum;
    };
    for (int e = threadIdx.x; e < (R / WU) * RB * M; e += blockDim.x) {
        const int rbi = e / (RB * M), rm = e % (RB * M), r = rm / M, m = rm % M;
        const int n = (rb0 / WU + rbi) * RB + r;
        if (n >= a.N) continue;
        if constexpr (GATED) {
            const float gsum = row_sum(2 * rbi, r, m), usum = row_sum(2 * rbi + 1, r, m);
            a.y[(long long)m * a.ldy + n] = __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul(gsum, usum)));
        } else {
            store_out(a, m, n, row_sum(rbi, r, m));
        }
    }
}

inline bool gemv_x_in_smem(int fmt, int K, int group, int M) {
    return gemv_smem_plan(fmt, K, group, M, true).total <= 227 * 1024;
}
inline size_t gemv_smem_bytes_impl(int fmt, int K, int group, int M) {
    if (gemv_is_mma(fmt)) return gemv_mma_smem_plan(fmt, K, group, M, gemv_mma_xmode(fmt, K, group, M)).total;
    return gemv_smem_plan(fmt, K, group, M, gemv_x_in_smem(fmt, K, group, M)).total;
}
inline int gemv_warps_impl(int fmt) {
    switch (fmt) {
        case UQ_INT4_SYM: return MmaCfg<UQ_INT4_SYM>::WARPS;
        case UQ_INT4_ASYM: return MmaCfg<UQ_INT4_ASYM>::WARPS;
        case UQ_INT2_ASYM: return MmaCfg<UQ_INT2_ASYM>::WARPS;
        case UQ_K4: return MmaCfg<UQ_K4>::WARPS;
        default: return GEMV_WARPS;
    }
}
inline size_t gemv_partials_floats_impl(int P, int M) { return (size_t)2 * P * RB * M; }

namespace gemv_detail {
template <int FMT, int M, bool XS>
cudaError_t launch_one(const GemvArgs& a, int grid, cudaStream_t st) {
    static bool configured[64] = {};   // the shared-memory opt-in, once per device
    const size_t smem = gemv_smem_plan_t<FMT>(a.K, a.group, M, XS).total;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gemv_kernel<FMT, M, XS>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    if (launch_overlap()) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(GEMV_WARPS * 32);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, gemv_kernel<FMT, M, XS>, a);
        if (e != cudaSuccess) return e;
    } else {
        gemv_kernel<FMT, M, XS><<<grid, GEMV_WARPS * 32, smem, st>>>(a);
    }
    return cudaGetLastError();
}
template <int FMT, int M>
cudaError_t launch_xs(const GemvArgs& a, int grid, cudaStream_t st) {
    if (gemv_x_in_smem(FMT, a.K, a.group, M)) return launch_one<FMT, M, true>(a, grid, st);
    return launch_one<FMT, M, false>(a, grid, st);
}
}  // namespace gemv_detail

namespace gemv_detail {
template <int FMT, int GB, int XM, bool GATED>
cudaError_t launch_mma(const GemvArgs& a, int grid, cudaStream_t st) {
    static bool configured[64] = {};
    const size_t smem = gemv_mma_smem_plan(FMT, a.K, a.group, a.M, XM).total;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gemv_mma_kernel<FMT, GB, XM, GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int threads = MmaCfg<FMT>::WARPS * 32;
    GemvArgs a2 = a;
    a2.overlap = launch_overlap() ? 1 : 0;
    if (a2.overlap) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, gemv_mma_kernel<FMT, GB, XM, GATED>, a2);
        if (e != cudaSuccess) return e;
    } else {
        gemv_mma_kernel<FMT, GB, XM, GATED><<<grid, threads, smem, st>>>(a2);
    }
    return cudaGetLastError();
}
template <int FMT, int GB, bool GATED>
cudaError_t launch_mma_xg(const GemvArgs& a, int grid, cudaStream_t st) {
    switch (gemv_mma_xmode(FMT, a.K, a.group, a.M)) {
        case MMA_X_SLICE: return launch_mma<FMT, GB, MMA_X_SLICE, GATED>(a, grid, st);
        case MMA_X_WHOLE: return launch_mma<FMT, GB, MMA_X_WHOLE, GATED>(a, grid, st);
        default: return launch_mma<FMT, GB, MMA_X_GLOBAL, GATED>(a, grid, st);
    }
}
template <int FMT, int GB>
cudaError_t launch_mma_xs(const GemvArgs& a, int grid, cudaStream_t st) {
    return a.gated ? launch_mma_xg<FMT, GB, true>(a, grid, st) : launch_mma_xg<FMT, GB, false>(a, grid, st);
}
}  // namespace gemv_detail

template <int FMT>
cudaError_t launch_gemv_fmt(const GemvArgs& a, int grid, cudaStream_t st) {
    if constexpr (FMT == UQ_INT4_SYM || FMT == UQ_INT4_ASYM || FMT == UQ_INT2_ASYM || FMT == UQ_K4) {
        const int gs = (FMT == UQ_K4) ? 32 : a.group;
        switch (gs) {
            case 32: return gemv_detail::launch_mma_xs<FMT, 2>(a, grid, st);
            case 64: if constexpr (FMT != UQ_K4) return gemv_detail::launch_mma_xs<FMT, 4>(a, grid, st);
                     return cudaErrorInvalidValue;
            case 128: if constexpr (FMT != UQ_K4) return gemv_detail::launch_mma_xs<FMT, 8>(a, grid, st);
                      return cudaErrorInvalidValue;
            default: return cudaErrorInvalidValue;
        }
    } else {
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
}

}  // namespace uq
