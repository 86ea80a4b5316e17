// uq_gemv.cuh -- small-M (M <= 8) fused dequantize + GEMV/GEMM, sm_103a.
//
// "Ultra LLM Engine", section "Fused Kernels": dequantized-weight GEMV for single-token
// decode and GEMM for batched decode.  Decode is bound by streaming the packed weights from
// HBM once; on this GPU the arithmetic of a CUDA-core dot product (unpack, widen, FMA: about
// three issue slots per 4-bit weight) cannot keep up with HBM, so the 4-bit and 2-bit formats
// run on warp-level tensor instructions:
//
//  * The packed plane is in mma.m16n8k16 A-fragment order: one 16-byte shared-memory load per
//    lane, a shift and a lop3 per register (magic exponent: bf16 0x4300 | code = 128 + code)
//    give the A fragments, and mma.sync (bf16 x bf16 -> fp32) does the multiply-accumulate and
//    the reduction over the 16-wide k block in one instruction; the M <= 8 activation rows are
//    the instruction's N = 8, so every M <= 8 costs the same.  Per scaling group the fp32 group
//    sum is folded as  s * (sum x*(128 + q) - (128 + z) * sum x),  in rounds of 8 groups: each
//    pair of groups folded from zero, then  tile += (p0 + p1) + (p2 + p3).  With one row of x the
//    round's 8 groups ride in the instruction's 8 columns instead (zeros in the B fragments of the
//    other groups' blocks), so the fold costs a lane 2 groups instead of 8: the same operations on
//    the same values in the same order, so a row's result is the same alone and in a batch.
//  * Work is the list of tiles (16 rows x 8 KB of codes) in k-major order.  Either every CTA owns
//    whole 16-row blocks (partial sums of each tile in shared memory, summed per row in k order
//    after a CTA barrier: no second launch), or CTAs own equal contiguous ranges of all tiles
//    (stream-K) and store each tile's partial sums in global memory for gemv_split_reduce, a
//    second launch that sums each row over its k tiles in k order.  Both orders are fixed, so
//    results are bit-reproducible, and a row's result is the same for either split and any M.
//  * gemv_mma_kernel (every format at M = 1..8, except the case below): one CTA per SM, a copy
//    warp feeding 12 compute warps through one ring of tile pairs (one 16 KB bulk copy per pair)
//    in nearly all of shared memory; x whole in shared memory (one row of it with the groups as
//    columns) or read through L1; the sums of x over each scaling group in a table formed once
//    per CTA.  INT8: the stored byte q + 128 =
//    16 hi + lo, its two nibbles through the same bf16 magic, two mma chains per block, sum q x =
//    16 D_hi + D_lo - 2304 sum x.  NF4: each codebook value c[q] as hi = bf16(c[q]) and lo =
//    bf16(c[q] - hi) (16 significant bits) from a 16-entry shared table, two mma chains per block.
//  * gemv_warp_kernel (INT4_SYM, INT4_ASYM at M = 1): the same per-tile arithmetic on per-warp
//    rings of two stages (16-byte cp.async by each warp's own lanes) and double-buffered slices
//    of x, two CTAs per SM.  Its launches are short, and two ~111 KB CTAs per SM let the next
//    launch on the stream start streaming while the current one finishes; measured faster there.
//    Both kernels form the sums of x in the same order, so they give the same rows.
//    With launch overlap both request their first weights before waiting for the previous
//    kernel on the stream (the weights are constant).
#pragma once
#include "uq_kernels.h"

namespace uq {

template <int FMT> struct GemvFmt {
    static constexpr int BITS = fmt_bits(FMT);
    static constexpr int KT = fmt_kt(FMT);
    static constexpr int KC = fmt_kc(FMT);
    static constexpr int BPC = KC / 16;                            // 16-wide k blocks per chunk
    static constexpr bool MMA = (FMT == UQ_INT4_SYM || FMT == UQ_INT4_ASYM || FMT == UQ_K4 || FMT == UQ_INT2_ASYM ||
                                 FMT == UQ_INT8_SYM || FMT == UQ_NF4);
    static constexpr int GT_MAX = KT / 32;                         // groups per tile row at group 32
};

// Stage geometry: a stage is one tile's codes followed by its rows' metadata, MW 32-bit words per
// row: scales (+1 word for a misaligned start), then zeros, each rounded up to 4 words so 16-byte
// copies land 16-byte aligned.  GT = groups per tile row the stage must hold (0: as many as the
// smallest group, 32, gives).  K4 rows hold their 16-byte super-block records.
template <int FMT, int GT = 0> struct MetaGeom {
    static constexpr int GTM = GT ? GT : GemvFmt<FMT>::GT_MAX;
    static constexpr int SW = (FMT == UQ_K4) ? 16 : (GTM / 2 + 1 + 3) / 4 * 4;
    static constexpr int ZW = (FMT == UQ_INT4_ASYM) ? (GTM / 8 + 1 + 3) / 4 * 4
                            : (FMT == UQ_INT2_ASYM ? (GTM / 2 + 1 + 3) / 4 * 4 : 0);
    static constexpr int MW = SW + ZW;
    static constexpr int META_BYTES = (RB * MW * 4 + 15) / 16 * 16;
    static constexpr int STAGE_BYTES = TILE_BYTES + META_BYTES;
};

// shared-memory offsets of a GEMV launch (the per-warp-ring kernels); identical on host and device
struct GemvSmem {
    size_t bars, lut, sx, ps, x, zr, total;
};

namespace {

__device__ __forceinline__ long long range_begin(int w, long long T, int P) { return (long long)w * T / P; }

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

// D += A * B for one 16 x 8 x 32 block: A unsigned 8-bit (the stored codes), B signed 8-bit (x codes),
// exact 32-bit integer accumulation
__device__ __forceinline__ void mma_u8s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

// Copy the metadata of tile (nb, kb)'s rows (scales, zero points or K4 records) into md, laid out
// as MetaGeom<FMT, GEO>, with cp.async by all lanes (not committed or counted here).  GTC: the
// groups per tile row when the caller knows them at compile time (0: mc.GT at run time).
template <int FMT, int GTC = 0, int GEO = 0>
__device__ __forceinline__ void issue_meta(const GemvArgs& a, const GemvSrc& w, const MetaConst& mc, int nb, int kb,
                                           uint32_t* md, int lane) {
    using F = MetaGeom<FMT, GEO>;
    const int n0 = nb * RB;
    const int rows = (a.N - n0) < RB ? (a.N - n0) : RB;            // rows with metadata
    if constexpr (FMT == UQ_K4) {
        // 16-byte records: one per 256 k of the tile row that lies inside K
        const int sb0 = kb * (GemvFmt<FMT>::KT / 256);
        int recs = mc.S4 - sb0;
        if (recs > GemvFmt<FMT>::KT / 256) recs = GemvFmt<FMT>::KT / 256;
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
        const int perd = per > 0 ? per : 1;             // (no copies at all when per is 0)
        for (int e = lane; e < rows * per; e += 32) {
            const int r = e / perd, j = e % perd;
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
}

// Issue the copies of tile t into stage buffer `st` (its codes, then its metadata at st +
// TILE_BYTES; all lanes take part): 16-byte cp.async for the codes (512 contiguous bytes per warp
// instruction) and the metadata, in one cp.async group per lane that the issuing warp itself waits
// for (the per-warp-ring kernels).  GTC: the groups per tile row when the caller knows them at
// compile time (0: mc.GT at run time).
template <int FMT, int GTC = 0>
__device__ __forceinline__ void issue_tile(const GemvArgs& a, const GemvSrc& w, const Layout& L, const MetaConst& mc, int nb, int kb,
                                           uint8_t* st, int lane) {
    issue_meta<FMT, GTC>(a, w, mc, nb, kb, reinterpret_cast<uint32_t*>(st + TILE_BYTES), lane);
    const int bytes = (int)L.tile_bytes(kb);
    const uint8_t* src = w.wq + L.tile_offset(nb, kb) + lane * 16;
    uint8_t* dst = st + lane * 16;
    if (bytes == TILE_BYTES) {
#pragma unroll
        for (int q = 0; q < TILE_BYTES / 512; ++q) cp_async16(dst + q * 512, src + q * 512);
    } else {
        for (int off = 0; lane * 16 + off < bytes; off += 512) cp_async16(dst + off, src + off);
    }
    cp_async_commit_group();
}

// Pointers to row r's staged scales (fp16) and zero points for tile kb: the staged words start
// at the word holding the row's first group, so only the parity / low bits of its offset matter.
template <int FMT>
struct RowPtrs {
    const uint16_t* s;
    const uint8_t* z;
};
template <int FMT, int GEO = 0>
__device__ __forceinline__ RowPtrs<FMT> row_ptrs(const uint8_t* st, const MetaConst& mc, int r, int n, int kb) {
    using F = MetaGeom<FMT, GEO>;
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
    const uint8_t* row = st + TILE_BYTES + r * MetaGeom<UQ_K4>::MW * 4;
    const uint4 rec = *reinterpret_cast<const uint4*>(row + 16 * (li >> 3));
    const int j = li & 7;
    const uint64_t sc48 = (uint64_t)rec.y | ((uint64_t)(rec.z & 0xFFFFu) << 32);
    const uint64_t m48 = (uint64_t)(rec.z >> 16) | ((uint64_t)rec.w << 16);
    dsc = half_bits_f32((uint16_t)(rec.x & 0xFFFF)) * (float)((sc48 >> (6 * j)) & 63);
    dmm = half_bits_f32((uint16_t)(rec.x >> 16)) * (float)((m48 >> (6 * j)) & 63);
}

}  // namespace

// ------------------------------------------------------------------------------------------------
// 4-bit and 2-bit formats: the GEMV on mma.sync.  GB = 16-k blocks per scaling group (2, 4 or 8;
// K4 uses its 32-weight sub-blocks, GB = 2).  M (1..8) is a runtime value: the instruction always
// computes 8 columns, so the work per weight does not depend on it.
//
// One CTA per SM: a copy warp and MMA_CW compute warps around one ring.  A ring slot holds a pair
// of tiles, two consecutive k tiles of one row block (16 KB of codes, contiguous in the packed
// plane, plus both tiles' metadata).  The copy warp requests the CTA's pairs in order: one 16 KB
// bulk copy of the codes (lane 0) and the metadata by cp.async from all lanes, all counted on the
// slot's "full" mbarrier.  Compute warp w takes tile w & 1 of the pairs w / 2, w / 2 + P, ... for
// P tile-taking warp pairs (MMA_CW / 2, or fewer: gemv_mma_pairs) and hands the slot back on its
// "empty" mbarrier (two arrivals per pair).  Bulk copies of
// 16 KB keep an SM's share of HBM bandwidth streaming from a few copies in flight, where one warp
// of 16-byte cp.async keeps about one tile in flight; the shared ring holds every tile in flight
// once, so shared memory feeds 12 compute warps per SM instead of 8.
//
// Per 16 x 16 block of weights a lane issues its share of a 16-byte code load, four lop3 (three
// after a shift) to form the A fragment, one 8-byte load of x and the mma.  Per group: two fp32
// FMAs per accumulator with the group's scale and zero-point term, the latter using the group's
// sum of x from a table the CTA forms before its first tile (8-k segments in a fixed order, then a
// fixed shuffle tree: the same sums for every M, so a row's result does not depend on M), in the
// rounds of 8 groups described at the top of this file.
//
// Pair order is k-major: pair i of a range is (k tile pair i / R, row block i % R) for R row
// blocks.  Every tile's partial sums are stored (shared memory when the CTA owns whole row blocks,
// global memory otherwise) and summed over the k tiles in k order afterwards, so a row's result
// does not depend on how the work was split either.
constexpr int MMA_CW = 12;                  // compute warps per CTA (even: a warp keeps one half of its pairs)
constexpr int MMA_PMAX = 16;                // ring slots (tile pairs) at most
constexpr int MMA_TPC = 48;                 // tiles per CTA at most when it owns whole row blocks
constexpr int MMA_BAR_BYTES = (2 * MMA_PMAX + 1) * 8 + 64;   // mbarriers, then NF4's 16-entry table
constexpr int MMA_SMEM = 227 * 1024;        // dynamic shared memory of the CTA at most

// bytes per row of x in shared memory: 32 bytes of padding put the four rows a half-warp's 8-byte
// B-fragment loads touch into different banks
// (xb bytes per k: 2 for bf16 x, 1 for W4A8's int8 codes)
__host__ __device__ inline size_t gemv_mma_x_stride(int Kp, int xb = 2) { return (size_t)Kp * xb + 32; }

// Where the mma GEMV reads x (template parameter XM): MMA_X_WHOLE, the CTA's window of x (the k
// tiles its work touches: all of K when it owns whole row blocks, a few k tiles under the stream-K
// split) copied into shared memory once per CTA; MMA_X_GLOBAL, straight from global memory (through
// L1), when that window would leave the ring too few slots.
// MMA_X_ROW1: one row of x (M = 1, not gated, not A8) in shared memory as MMA_X_WHOLE, the groups
// of a round in the mma's columns.
constexpr int MMA_X_GLOBAL = 0, MMA_X_WHOLE = 1, MMA_X_ROW1 = 2;

// metadata bytes of one tile at this group size
template <int FMT>
__host__ __device__ inline int gemv_mma_meta_t(int gs) {
    constexpr int KT = fmt_kt(FMT);
    if (FMT == UQ_K4 || gs == 32) return MetaGeom<FMT, KT / 32>::META_BYTES;
    if (gs == 64) return MetaGeom<FMT, KT / 64>::META_BYTES;
    return MetaGeom<FMT, KT / 128>::META_BYTES;
}
__host__ __device__ inline int gemv_mma_meta(int fmt, int group) {
    switch (fmt) {
        case UQ_INT4_SYM: return gemv_mma_meta_t<UQ_INT4_SYM>(group);
        case UQ_INT4_ASYM: return gemv_mma_meta_t<UQ_INT4_ASYM>(group);
        case UQ_INT2_ASYM: return gemv_mma_meta_t<UQ_INT2_ASYM>(group);
        case UQ_INT8_SYM: return gemv_mma_meta_t<UQ_INT8_SYM>(group);
        case UQ_NF4: return gemv_mma_meta_t<UQ_NF4>(group);
        default: return gemv_mma_meta_t<UQ_K4>(32);
    }
}

// Groups in the CTA's table of x sums: those of every k tile when CTAs own whole row blocks (tpc >
// 0), else those of the k tiles a stream-K range of at most ceil(NB * KB2 / grid) consecutive
// k-major pairs can touch (at most ceil(range / NB) + 1 pairs of k tiles).
__host__ __device__ inline int gemv_mma_sx_groups(int fmt, int group, int NB, int KB, int grid, int tpc) {
    const int gs = fmt == UQ_K4 ? 32 : group;
    const int gpt = fmt_kt(fmt) / gs;
    long long span = KB;
    if (tpc == 0) {
        const long long P2 = (long long)NB * ((KB + 1) / 2);
        const long long per = (P2 + grid - 1) / grid;
        const long long touched = 2 * ((per + NB - 1) / NB + 1);
        if (touched < span) span = touched;
    }
    return (int)span * gpt;
}

// Shared memory: codes [S2][2][8 KB] | metadata [S2][2][meta] | full[S2], empty[S2] and x
// mbarriers, NF4's table | sums of x [groups][8] | partial sums [tiles of the CTA][16][8] (whole row blocks) |
// x (MMA_X_WHOLE) | zeros (MMA_X_WHOLE, one row of x).  S2 = the slots that fit beside the rest (at most MMA_PMAX).  Identical on
// host and device.
struct MmaSmem {
    size_t meta, bars, sx, ps, x, zr, total;
    int S2, mb;                                     // slots, metadata bytes per tile
};
// one row of x in shared memory also takes 256 bytes of zeros (B fragments of the other groups'
// columns), 32 bytes past a 128-byte boundary so a load's x lanes and zero lanes hit different banks
__host__ __device__ inline bool gemv_mma_colmode(int M, int xm) { return M == 1 && xm == MMA_X_ROW1; }
// offsets for S2 slots (multiplications and additions only: the kernel forms them per launch)
__host__ __device__ inline MmaSmem gemv_mma_offsets(int S2, int mb, int sxg, int tpc, int M, int xk, int xm, int xb = 2) {
    MmaSmem p;
    p.S2 = S2;
    p.mb = mb;
    p.meta = (size_t)S2 * 2 * TILE_BYTES;
    p.bars = p.meta + (size_t)S2 * 2 * mb;
    p.sx = (p.bars + (size_t)MMA_BAR_BYTES + 15) / 16 * 16;
    p.ps = p.sx + (size_t)sxg * 8 * 4;
    p.x = (p.ps + (size_t)tpc * RB * 8 * 4 + 127) / 128 * 128;
    p.total = p.x + (xm != MMA_X_GLOBAL ? (size_t)M * gemv_mma_x_stride(xk, xb) : 0);
    p.zr = 0;
    if (gemv_mma_colmode(M, xm)) {
        p.zr = (p.total + 127) / 128 * 128 + 32;
        p.total = p.zr + 256;
    }
    return p;
}
__host__ __device__ inline MmaSmem gemv_mma_smem(int fmt, int K, int group, int M, int sxg, int tpc, int xm, int xb = 2) {
    const int mb = gemv_mma_meta(fmt, group);
    const int slot = 2 * (TILE_BYTES + mb);
    const int gpt = fmt_kt(fmt) / (fmt == UQ_K4 ? 32 : group);
    const int xk = sxg / gpt * fmt_kt(fmt);                         // k extent of a CTA's window of x
    (void)K;
    const size_t bars = (size_t)MMA_BAR_BYTES;
    const size_t xbytes = (xm != MMA_X_GLOBAL ? (size_t)M * gemv_mma_x_stride(xk, xb) : 0) +
                          (gemv_mma_colmode(M, xm) ? 127 + 32 + 256 : 0);
    const size_t rest = bars + 16 + (size_t)sxg * 8 * 4 + (size_t)tpc * RB * 8 * 4 + 128 + xbytes;   // + alignment
    long long S2 = ((long long)MMA_SMEM - (long long)rest) / slot;
    if (S2 > MMA_PMAX) S2 = MMA_PMAX;
    if (S2 < 0) S2 = 0;
    return gemv_mma_offsets((int)S2, mb, sxg, tpc, M, xk, xm, xb);
}
// x in shared memory when that leaves the ring 2 slots beyond those the compute warps hold
// (measured: 8 rows of x through L1 cost more than a shallower ring)
// (row1: MMA_X_ROW1 allowed, for one row of x when it fits as well)
__host__ __device__ inline int gemv_mma_xmode(int fmt, int K, int group, int M, int sxg, int tpc, int xb = 2,
                                              bool row1 = false) {
    if (gemv_mma_smem(fmt, K, group, M, sxg, tpc, MMA_X_WHOLE, xb).S2 < MMA_CW / 2 + 2) return MMA_X_GLOBAL;
    if (row1 && M == 1 && gemv_mma_smem(fmt, K, group, M, sxg, tpc, MMA_X_ROW1, xb).S2 >= MMA_CW / 2 + 2)
        return MMA_X_ROW1;
    return MMA_X_WHOLE;
}

// Pairs of compute warps that take tiles (the rest only help form the table of x sums).  Measured
// (bench, 4 against 6 pairs, same box): INT8 8192^2 at M = 1 3060 / 3012 GB/s, the INT4 sweep at
// M = 8 2433 / 2394 and M = 2, 4 level; NF4 1672 / 1719, K4 at M = 1 and 8 2798 / 2830 and
// 1672 / 1747, W4A8 1911 / 2016.  With fewer pairs each holds more of the ring (3 slots of 12
// instead of 2), which pays where a tile's compute is light; the heavier unpacks want the warps.
__host__ __device__ inline int gemv_mma_pairs(int fmt, bool a8) {
    return !a8 && (fmt == UQ_INT4_SYM || fmt == UQ_INT4_ASYM || fmt == UQ_INT8_SYM) ? 4 : MMA_CW / 2;
}

__device__ __forceinline__ float bf16_pair_sum(uint32_t w) {
    return __uint_as_float(w << 16) + __uint_as_float(w & 0xFFFF0000u);
}
__device__ __forceinline__ void compute_warps_sync() {
    asm volatile("bar.sync 1, %0;" :: "n"(MMA_CW * 32) : "memory");
}

// GATED: the gated projection in one launch.  The work list interleaves the gate and up weights' row
// blocks (work row block 2j = gate row block j, 2j + 1 = up row block j), every CTA owns whole pairs,
// and the per-row reduction forms h = silu(g) * u (or the second pass does, for the stream-K split).
// A8: W4A8 / W8A8 (INT4_SYM, INT4_ASYM, INT8_SYM): x is the int8 codes of a.xq (1 byte per k, each
// 32 k in the integer mma's B fragment order), the table holds the quantizer's integer code sums,
// the group step is mma.m16n8k32 (u8 x s8 -> s32) on the stored codes as bytes, and each tile's
// partial sums are scaled by the row's s_x.
template <int FMT, int GB, int XM, bool GATED, bool A8 = false>
__global__ void __launch_bounds__((MMA_CW + 1) * 32, 1) gemv_mma_kernel(const GemvArgs a) {
    using F = GemvFmt<FMT>;
    constexpr int KT = F::KT, CW = MMA_CW, PW = MMA_CW / 2;
    static_assert(MMA_CW % 2 == 0, "compute warps come in pairs");
    static_assert(!A8 || ((FMT == UQ_INT4_SYM || FMT == UQ_INT4_ASYM || FMT == UQ_INT8_SYM) && !GATED),
                  "the integer path takes INT4_SYM, INT4_ASYM and INT8_SYM, not gated");
    constexpr int XBY = A8 ? 1 : 2;                                 // bytes of x per k
    constexpr int GS = GB * 16;                                     // k per scaling group
    constexpr int GPT = KT / GS;                                    // groups per full tile row
    constexpr int MB = MetaGeom<FMT, GPT>::META_BYTES;              // metadata bytes per tile
    constexpr int WPG = (FMT == UQ_INT2_ASYM) ? GB / 2 : (FMT == UQ_INT8_SYM ? 2 * GB : GB);   // code words per lane per group
    constexpr int BPCH = F::BPC;                                    // 16-k blocks per 512-byte chunk
    constexpr bool XS = XM != MMA_X_GLOBAL;                        // x in shared memory
    constexpr bool COL = XM == MMA_X_ROW1;                          // one row of x, groups as columns
    static_assert(!COL || (!A8 && !GATED), "the column scheme takes one plain row of x");
    extern __shared__ __align__(128) uint8_t smem[];
    const int M = a.M;
    const int tpc = a.cta_rows;                                     // > 0: CTAs own whole row blocks
    const bool cta_rows = tpc > 0;
    const Layout L(a.N, a.K, FMT);
    const int sxg = a.sx_groups;
    const int XK = sxg / GPT * KT;                                  // k extent of the CTA's window of x
    const MmaSmem plan = gemv_mma_offsets(a.ring_slots, MB, sxg, tpc, M, XK, XM, XBY);
    const int S2 = plan.S2;
    uint8_t* ring = smem;                                           // codes: slot s, tile h at (2s + h) * 8 KB
    uint8_t* metas = smem + plan.meta;                              // metadata: slot s, tile h at (2s + h) * MB
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
    uint64_t* empty = full + S2;
    uint64_t* xbar = full + 2 * S2;
    uint32_t* nlut = reinterpret_cast<uint32_t*>(smem + plan.bars + (2 * MMA_PMAX + 1) * 8);   // NF4: (hi | lo << 16)
    float* sxt = reinterpret_cast<float*>(smem + plan.sx);
    float* cpart = reinterpret_cast<float*>(smem + plan.ps);
    uint8_t* xs = smem + plan.x;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    // COL: the groups of a round of 8 ride in the mma's columns (gemv_warp_kernel's scheme), and the
    // scales fold once per group and row instead of once per group, row and lane
    const uint8_t* xz = smem + plan.zr + 8 * c;                     // zeros (COL)

    // Work split over pairs of k tiles (KB2 per row block; when KB is odd the last pair holds one
    // tile): whole row blocks [rb0, rb0 + R) per CTA (gated: gate / up pairs), or the stream-K range
    // [p0, p1) of all NB * KB2 pairs.  Local pair pl is pair p0 + pl of the k-major order over R row
    // blocks: k tiles 2 ((p0 + pl) / R) + {0, 1}, row block rb0 + (p0 + pl) % R (R = NB for
    // stream-K).  Local tile li = 2 pl + h.
    // (32-bit arithmetic: the host plans no launch with 2^31 pairs or more; the divisions here sit
    // on the copy warp's path to its first request)
    constexpr int WU = GATED ? 2 : 1;
    const unsigned b = blockIdx.x, nctas = gridDim.x;
    const unsigned NBU = (unsigned)a.NB / WU;
    const unsigned KB2 = ((unsigned)a.KB + 1) / 2;
    int rb0 = 0, R = a.NB;
    unsigned p0 = 0, npl;
    if (cta_rows) {                              // the first NBU % nctas CTAs own one row block more
        const unsigned q = NBU / nctas, r = NBU - q * nctas;
        rb0 = WU * (int)(b * q + (b < r ? b : r));
        R = WU * (int)(q + (b < r ? 1u : 0u));
        npl = (unsigned)R * KB2;
    } else {                                     // the first P2 % nctas CTAs take one pair more
        const unsigned P2 = (unsigned)a.NB * KB2;
        const unsigned q = P2 / nctas, r = P2 - q * nctas;
        p0 = b * q + (b < r ? b : r);
        npl = q + (b < r ? 1u : 0u);
    }
    // pair p0 + i as (k tile pair, row block index): one division here, increments afterwards
    const int kp0 = (int)(p0 / (unsigned)R), rp0 = (int)(p0 - (unsigned)kp0 * (unsigned)R);
    const int kb_first = npl > 0 ? 2 * kp0 : 0;
    int kb_last = npl > 0 ? 2 * (int)((p0 + npl - 1) / (unsigned)R) + 1 : -1;
    if (kb_last > a.KB - 1) kb_last = a.KB - 1;
    const int nsx = (kb_last - kb_first + 1) * GPT;                 // table groups this CTA uses
    // pairs of compute warps that take tiles (the others only help form the table of x sums); a CTA
    // with no more pairs than PW gives each pair to its own warp pair
    const int PWn = (a.mma_pairs > 0 && a.mma_pairs < PW && (int)npl > PW) ? a.mma_pairs : PW;
    const bool bad = (cta_rows && 2 * (int)npl > tpc) || nsx > sxg || S2 <= PWn || R <= 0 ||
                     (COL && M != 1);                               // never planned
    if (bad) {
        if (threadIdx.x == 0) atomicOr(a.fault, FAULT_GEMV_SPLIT);
        return;
    }
    const int G_all = a.K / GS;                                     // scaling groups per row
    const size_t xstride = gemv_mma_x_stride(XK, XBY);

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == CW) {
        // ---- copy warp: initializes the mbarriers and signals named barrier 2 without waiting, then
        // requests the CTA's pairs in order into the ring (per pair the codes, then the metadata),
        // the first ring's worth at once and then pair by pair as slots come back.  The weights are
        // constant, so it does not wait for the previous kernel on the stream.
        if (lane == 0) {
            for (int s = 0; s < S2; ++s) {
                mbar_init(&full[s], 33);                            // 32 lanes' metadata + the codes' expect_tx
                mbar_init(&empty[s], 2);                            // the pair's two compute warps
            }
            mbar_init(xbar, 1);
            fence_barrier_init();
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" :: "n"((CW + 1) * 32) : "memory");
        const GemvSrc src_gate{a.wq, a.scales, a.zc}, src_up{a.wq2, a.scales2, a.zc2};
        // the codes of pair (k tile pair kp, row block index rb) into slot s (lane 0)
        auto codes = [&](int kp, int rb, int s) {
            const int nbw = rb0 + rb, nb = GATED ? nbw >> 1 : nbw;
            const uint8_t* wq = (GATED && (nbw & 1)) ? a.wq2 : a.wq;
            const int kb0 = 2 * kp;
            // tile kb0 is whole when kb0 + 1 exists (only the last k tile can be narrower)
            const uint32_t bytes = kb0 + 1 < a.KB ? (uint32_t)(TILE_BYTES + L.tile_bytes(kb0 + 1)) : (uint32_t)L.tile_bytes(kb0);
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&full[s], bytes);
            bulk_g2s(ring + (size_t)s * 2 * TILE_BYTES, wq + L.tile_offset(nb, kb0), bytes, &full[s]);
        };
        const int first = (int)npl < S2 ? (int)npl : S2;
        MetaConst mc;
        mc.G = a.K / a.group;
        mc.GT = KT / a.group;
        mc.ZB = (mc.G + 1) >> 1;
        mc.S4 = a.K / 256;
        mc.aligned = (a.K % (8 * a.group)) == 0 && (mc.GT % 8) == 0;
        // the metadata of pair (kp, rb) into slot s, each lane's copies arriving on its full barrier
        auto meta = [&](int kp, int rb, int s) {
            const int nbw = rb0 + rb, nb = GATED ? nbw >> 1 : nbw;
            const GemvSrc& src = (GATED && (nbw & 1)) ? src_up : src_gate;
            const int kb0 = 2 * kp;
            uint32_t* md = reinterpret_cast<uint32_t*>(metas + (size_t)s * 2 * MB);
            issue_meta<FMT, GPT, GPT>(a, src, mc, nb, kb0, md, lane);
            if (kb0 + 1 < a.KB) issue_meta<FMT, GPT, GPT>(a, src, mc, nb, kb0 + 1, md + MB / 4, lane);
            cp_async_arrive_noinc(&full[s]);
        };
        int ikp = kp0, irb = rp0;
        for (int s = 0; s < first; ++s) {
            if (lane == 0) codes(ikp, irb, s);
            meta(ikp, irb, s);
            if (++irb == R) { irb = 0; ++ikp; }
        }
        int issued = first;
        int slot = 0;                                               // first < S2 only when npl == first
        uint32_t ph = 1;
        for (int pl = first; pl < (int)npl; ++pl) {
            // the slot's previous pair is done
            const bool ok = mbar_wait_bounded(&empty[slot], ph ^ 1u, a.fault, FAULT_GEMV_WAIT);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) codes(ikp, irb, slot);
            meta(ikp, irb, slot);
            ++issued;
            if (++irb == R) { irb = 0; ++ikp; }
            if (++slot == S2) { slot = 0; ph ^= 1u; }
        }
        // nothing the warp requested may land after the CTA has left: its own cp.async, then the
        // last pairs' bulk copies (their full phases complete)
        asm volatile("cp.async.wait_all;" ::: "memory");
        for (int q = (issued > S2 ? issued - S2 : 0); q < issued; ++q)
            mbar_wait_bounded(&full[q % S2], (uint32_t)((q / S2) & 1), a.fault, FAULT_GEMV_WAIT);
        return;
    }

    // ---- compute warps.  x may be written by the previous kernel on the stream.
    MetaConst mc;
    mc.G = a.K / a.group;
    mc.GT = KT / a.group;
    mc.ZB = (mc.G + 1) >> 1;
    mc.S4 = a.K / 256;
    mc.aligned = (a.K % (8 * a.group)) == 0 && (mc.GT % 8) == 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("bar.sync 2, %0;" :: "n"((CW + 1) * 32) : "memory");   // the mbarriers are initialized
    if constexpr (XS) {
        // the CTA's window of x: k tiles kb_first .. kb_last of every row (the tiles' groups lie
        // inside K, so nothing past K is read)
        if (threadIdx.x == 0) {
            const int k0 = kb_first * KT;
            const int kend = A8 ? a.Kpq : a.K;                      // (the codes are zero-padded to Kpq)
            const int k1 = (kb_last + 1) * KT < kend ? (kb_last + 1) * KT : kend;
            mbar_arrive_expect_tx(xbar, (uint32_t)(M * (k1 - k0) * XBY));
            for (int m = 0; m < M; ++m) {
                const void* src = A8 ? (const void*)(a.xq + (long long)m * a.Kpq + k0)
                                     : (const void*)(a.x + (long long)m * a.ldx + k0);
                bulk_g2s(xs + m * xstride, src, (uint32_t)((k1 - k0) * XBY), xbar);
            }
        }
    }
    {
        // table of x sums: entry (group gl of k tiles kb_first.., column m) = the sum of row m of x
        // over the group.  A warp task is one row of x over one k tile: lane l adds k = KL l .. KL l
        // + KL - 1 in order (a bf16 pair at a time), then a group's GS / KL lanes combine by a
        // shuffle tree (or a lane's KL k hold KL / GS groups).  This is the order gemv_warp_kernel
        // forms its sums in, so the two kernels give the same sums (and rows of y) for any M.  Each
        // round issues its tasks' loads before any sum (a load's first use would stall the next).
        // Columns m >= M are zero (their products are never stored).
        if constexpr (A8) {
            // the quantizer's per-group code sums (exact integers, below 2^24 in magnitude)
            const int Gq = (a.Kpq + GS - 1) / GS;
            for (int e = threadIdx.x; e < M * nsx; e += CW * 32) {
                const int m = e / nsx, gl = e - m * nsx, gi = kb_first * GPT + gl;
                if (gi < G_all) sxt[gl * 8 + m] = (float)__ldg(a.sxl + (long long)m * Gq + gi);
            }
        } else {
            constexpr int KL = KT / 32;                                 // k per lane
            constexpr int NV = KL / 8;                                  // 16-byte loads per lane and task
            constexpr int TU = NV >= 8 ? 1 : 8 / NV;                    // tasks per warp per round
            constexpr int NGL = (KL / GS) > 1 ? (KL / GS) : 1;          // groups within a lane's k
            const int nkt = kb_last - kb_first + 1;
            const int ntask = M * nkt;
            for (int tb = warp; tb < ntask; tb += TU * CW) {
                uint4 w[TU][NV];
#pragma unroll
                for (int u = 0; u < TU; ++u) {
                    const int t = tb + u * CW;
                    const int m = t / nkt, kt = kb_first + (t - m * nkt);   // warp-uniform
                    const int k0 = kt * KT + lane * KL;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        w[u][v] = make_uint4(0u, 0u, 0u, 0u);
                        if (t < ntask && k0 + 8 * v < a.K) w[u][v] = ldg_nc_v4(a.x + (long long)m * a.ldx + k0 + 8 * v);
                    }
                }
#pragma unroll
                for (int u = 0; u < TU; ++u) {
                    const int t = tb + u * CW;
                    const int m = t / nkt, ktl = t - m * nkt;
                    float gsum[NGL];
#pragma unroll
                    for (int q = 0; q < NGL; ++q) gsum[q] = 0.f;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        const uint32_t wv4[4] = {w[u][v].x, w[u][v].y, w[u][v].z, w[u][v].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const int q = (NGL > 1) ? (v * 8 + 2 * h) / GS : 0;
                            gsum[q] += bf16_pair_sum(wv4[h]);
                        }
                    }
                    if constexpr (GS >= KL) {
#pragma unroll
                        for (int o = 1; o < GS / KL; o <<= 1) gsum[0] += __shfl_xor_sync(0xffffffffu, gsum[0], o);
                        const int gl = ktl * GPT + lane / (GS / KL);
                        if (t < ntask && (lane & (GS / KL - 1)) == 0 && kb_first * GPT + gl < G_all) sxt[gl * 8 + m] = gsum[0];
                    } else {
#pragma unroll
                        for (int q = 0; q < NGL; ++q) {
                            const int gl = ktl * GPT + lane * NGL + q;
                            if (t < ntask && kb_first * GPT + gl < G_all) sxt[gl * 8 + m] = gsum[q];
                        }
                    }
                }
            }
        }
        for (int e = threadIdx.x; e < nsx * 8; e += CW * 32)
            if ((e & 7) >= M) sxt[e] = 0.f;
        if (COL && threadIdx.x < 64) reinterpret_cast<uint32_t*>(smem + plan.zr)[threadIdx.x] = 0u;
    }
    if constexpr (FMT == UQ_NF4) {
        // the codebook value c[q] as hi = bf16(c[q]) and lo = bf16(c[q] - hi): hi + lo carries 16
        // significant bits of c[q] (relative error below 2^-16); two mma chains multiply x by both
        if (threadIdx.x < 16) {
            const float cq = reinterpret_cast<const float*>(a.zc)[threadIdx.x];
            const __nv_bfloat16 hi = __float2bfloat16_rn(cq);
            const __nv_bfloat16 lo = __float2bfloat16_rn(cq - __bfloat162float(hi));
            nlut[threadIdx.x] = (uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(lo) << 16);
        }
    }
    compute_warps_sync();                                           // the table and x padding are written
    bool xok = true;
    if constexpr (XS) xok = mbar_wait_bounded(xbar, 0, a.fault, FAULT_GEMV_WAIT);
    const int npl_w = __all_sync(0xffffffffu, xok) ? (int)npl : 0;

    float acc[4] = {0.f, 0.f, 0.f, 0.f};        // rows g + 8j, columns 2c + e
    const int mrow = g < M ? g : M - 1;          // B rows beyond M repeat a real row; their D columns are unused
    const uint16_t* xgrow = a.x + (long long)mrow * a.ldx + 4 * c;
    const uint8_t* xrow = xs + mrow * xstride + 8 * c;
    float sxm[2] = {1.f, 1.f};                   // A8: the scales of x of columns 2c, 2c + 1
    const int8_t* xg8row = nullptr;              // A8: this lane's x codes in global memory
    if constexpr (A8) {
#pragma unroll
        for (int e = 0; e < 2; ++e) sxm[e] = 2 * c + e < M ? __ldg(a.sxq + 2 * c + e) : 0.f;
        xg8row = a.xq + (long long)mrow * a.Kpq + 8 * c;
    }
    // this warp's tiles: tile hh of the pairs pl = warp / 2, warp / 2 + PWn, ...; pair coordinates
    // advanced by (PWn / R, PWn % R)
    const int hh = warp & 1;
    const int dq = PWn / R, dr = PWn % R;
    int ckp = kp0, crb = rp0 + (warp >> 1);      // pair p0 + warp / 2 (warp / 2 < PW: a few steps at most)
    while (crb >= R) { crb -= R; ++ckp; }
    int slot = warp >> 1;                        // pl % S2 (PWn < S2: one wrap per step at most)
    uint32_t ph = 0;                             // (pl / S2) & 1
    for (int pl = (warp >> 1) < PWn ? warp >> 1 : npl_w; pl < npl_w; pl += PWn) {
        const int kb = 2 * ckp + hh, nbw = rb0 + crb, nb = GATED ? nbw >> 1 : nbw;
        ckp += dq;
        crb += dr;
        if (crb >= R) { crb -= R; ++ckp; }
        const bool ok = mbar_wait_bounded(&full[slot], ph, a.fault, FAULT_GEMV_WAIT);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (kb < a.KB) {                         // (the second tile of a pair at an odd KB's end does not exist)
            const int n0 = nb * RB;
            const int gi0 = kb * GPT;
            const int ng = (G_all - gi0) < GPT ? (G_all - gi0) : GPT;   // groups of the tile inside K
            const float* sxc = sxt + (gi0 - kb_first * GPT) * 8;      // the tile's groups, column 0
            const float* sxk = sxc + 2 * c;
            const uint8_t* xt = xrow + (size_t)(kb - kb_first) * KT * XBY;
            const uint16_t* xgt = xgrow + (long long)kb * KT;
            const int8_t* xg8 = A8 ? xg8row + (long long)kb * KT : nullptr;
            const uint8_t* st = ring + (size_t)(2 * slot + hh) * TILE_BYTES;
            // the tile's metadata, addressed as if it followed the codes (row_ptrs / row_meta_k4 add
            // TILE_BYTES; the address stays inside the ring)
            const uint8_t* sm = metas + (size_t)(2 * slot + hh) * MB - TILE_BYTES;
            RowPtrs<FMT> rp[2];
            if constexpr (FMT != UQ_K4) {
                rp[0] = row_ptrs<FMT, GPT>(sm, mc, g, n0 + g, kb);
                rp[1] = row_ptrs<FMT, GPT>(sm, mc, g + 8, n0 + g + 8, kb);
            }

            // A8: one group's exact integer products, folded into p (= acc)
            auto group_a8 = [&](const int gg, float (&p)[4]) {
                if constexpr (A8) {
                    // the group's exact integer sums of (stored code) x (x code) per row and column: GB / 2
                    // instructions of m16n8k32, each over two 16-k blocks (A: the two rows' codes as bytes,
                    // w & 0x0F0F0F0F and (w >> 4) & 0x0F0F0F0F for 4-bit; INT8 words are already bytes)
                    int di[4] = {0, 0, 0, 0};
#pragma unroll
                    for (int t = 0; t < GB / 2; ++t) {
                        const int blk = gg * GB + 2 * t;
                        uint32_t a0, a1, a2, a3;
                        if constexpr (FMT == UQ_INT8_SYM) {
                            const uint4 v = *reinterpret_cast<const uint4*>(st + (blk / BPCH) * CHUNK + lane * 16);
                            a0 = v.x; a1 = v.y; a2 = v.z; a3 = v.w;
                        } else {
                            const uint2 v = *reinterpret_cast<const uint2*>(st + (blk / BPCH) * CHUNK + lane * 16 +
                                                                            (blk % BPCH) * 4);
                            a0 = v.x & 0x0F0F0F0Fu;                 // row g:     k, k+2, k+1, k+3
                            a1 = (v.x >> 4) & 0x0F0F0F0Fu;          // row g + 8: the same order
                            a2 = v.y & 0x0F0F0F0Fu;
                            a3 = (v.y >> 4) & 0x0F0F0F0Fu;
                        }
                        uint2 bv;                                   // the pair's x codes of column g, in B order
                        if constexpr (XS) bv = *reinterpret_cast<const uint2*>(xt + blk * 16);
                        else bv = ldg_nc_v2(xg8 + blk * 16);
                        mma_u8s8(di, a0, a1, a2, a3, bv.x, bv.y);
                    }
                    // fold: acc += s * (D - zc * SX), SX the group's code sum of the column, zc the stored
                    // code's offset (8 for INT4_SYM, z for INT4_ASYM, 128 for INT8_SYM)
                    const float2 sxv = *reinterpret_cast<const float2*>(sxk + gg * 8);
                    const int sx0 = (int)sxv.x, sx1 = (int)sxv.y;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float sc, zcf;
                        row_meta<FMT>(rp[j], gg, sc, zcf);
                        const int zc = (FMT == UQ_INT8_SYM) ? 128 : (int)zcf - 128;
                        p[2 * j] = fmaf(sc, (float)(di[2 * j] - zc * sx0), p[2 * j]);
                        p[2 * j + 1] = fmaf(sc, (float)(di[2 * j + 1] - zc * sx1), p[2 * j + 1]);
                    }
                    return;
                }
            };
            // one group's products into the chains dd
            auto group_mma = [&](const int gg, float (&dd)[2][4], const bool first, const bool col) {
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
                    } else if constexpr (WPG == 16) {                  // INT8 at 128-k groups: 4 chunks
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 v = *reinterpret_cast<const uint4*>(cp + q * CHUNK);
                            wv[4 * q] = v.x; wv[4 * q + 1] = v.y; wv[4 * q + 2] = v.z; wv[4 * q + 3] = v.w;
                        }
                    } else if constexpr (WPG == 2) {
                        const uint2 v = *reinterpret_cast<const uint2*>(cp);
                        wv[0] = v.x; wv[1] = v.y;
                    } else {
                        wv[0] = *reinterpret_cast<const uint32_t*>(cp);
                    }
                }
                // B fragments: x at k = 16 blk + 4c .. +3 of row mrow (8 bytes per block); every block
                // of a group inside K lies inside K (K is a multiple of the group).  `col`: one row of
                // x, column g carrying group 8r + g of the round (zeros for the other groups' blocks)
                uint32_t bx[GB], by[GB];
                const uint8_t* xg = xt + gg * GB * 32;
                if (col && g != (gg & 7)) xg = xz;
#pragma unroll
                for (int j = 0; j < GB; ++j) {
                    uint2 v;
                    if constexpr (XS) v = *reinterpret_cast<const uint2*>(xg + j * 32);
                    else v = ldg_nc_v2(xgt + (gg * GB + j) * 16);
                    if constexpr (FMT == UQ_INT8_SYM) {
                        // an INT8 word holds k 4c .. 4c + 3 of one row and its nibble pairs come out as
                        // (4c, 4c + 2) and (4c + 1, 4c + 3): x paired the same way
                        bx[j] = __byte_perm(v.x, v.y, 0x5410);
                        by[j] = __byte_perm(v.x, v.y, 0x7632);
                    } else {
                        bx[j] = v.x; by[j] = v.y;
                    }
                }
                // the group's sum of (128 + q) x, in two chains (even / odd blocks); INT8: the sums
                // over the stored bytes' high and low nibbles, (128 + hi) x and (128 + lo) x; NF4: the
                // sums over the codebook values' hi and lo parts (no offset: zc = 0).  The chains start
                // from zero at the group (or round) when `first`.
#pragma unroll
                for (int j = 0; j < GB; ++j) {
                    uint32_t a0, a1, a2, a3;
                    if constexpr (FMT == UQ_INT8_SYM) {
                        // chunk j / 2 holds blocks j & ~1, j | 1: words (block, row g) and (block, row g + 8)
                        const uint32_t wg = wv[4 * (j >> 1) + 2 * (j & 1)], wg8 = wv[4 * (j >> 1) + 2 * (j & 1) + 1];
                        const uint32_t h0 = nib_pair_lop3<1>(wg), h1 = nib_pair_lop3<1>(wg8);
                        const uint32_t h2 = nib_pair_lop3<3>(wg), h3 = nib_pair_lop3<3>(wg8);
                        a0 = nib_pair_lop3<0>(wg); a1 = nib_pair_lop3<0>(wg8);
                        a2 = nib_pair_lop3<2>(wg); a3 = nib_pair_lop3<2>(wg8);
                        if (first && j == 0) {
                            mma_bf16_zero(dd[0], a0, a1, a2, a3, bx[j], by[j]);
                            mma_bf16_zero(dd[1], h0, h1, h2, h3, bx[j], by[j]);
                        } else {
                            mma_bf16(dd[0], a0, a1, a2, a3, bx[j], by[j]);
                            mma_bf16(dd[1], h0, h1, h2, h3, bx[j], by[j]);
                        }
                        continue;
                    }
                    if constexpr (FMT == UQ_NF4) {
                        // pair P: the codes at bits 4P and 16 + 4P, their values from the table
                        const uint32_t wd = wv[j];
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int P = 0; P < 4; ++P) {
                            const uint32_t e = nlut[(wd >> (4 * P)) & 15u], o = nlut[(wd >> (16 + 4 * P)) & 15u];
                            hi[P] = __byte_perm(e, o, 0x5410);
                            lo[P] = __byte_perm(e, o, 0x7632);
                        }
                        if (first && j == 0) {
                            mma_bf16_zero(dd[0], hi[0], hi[1], hi[2], hi[3], bx[j], by[j]);
                            mma_bf16_zero(dd[1], lo[0], lo[1], lo[2], lo[3], bx[j], by[j]);
                        } else {
                            mma_bf16(dd[0], hi[0], hi[1], hi[2], hi[3], bx[j], by[j]);
                            mma_bf16(dd[1], lo[0], lo[1], lo[2], lo[3], bx[j], by[j]);
                        }
                        continue;
                    }
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
                    if (first && j < 2) mma_bf16_zero(dd[j & 1], a0, a1, a2, a3, bx[j], by[j]);
                    else mma_bf16(dd[j & 1], a0, a1, a2, a3, bx[j], by[j]);
                }
            };
            // p += the group's term from its chains: s * (D - zc * sum x) (K4: d sc D - (128 d sc +
            // dmin m) sum x), with the group's sums of x from the table
            auto fold = [&](const int gg, const float (&dd)[2][4], float (&p)[4]) {
                const float2 sxv = *reinterpret_cast<const float2*>(sxk + gg * 8);
                float d[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // INT8: the stored byte is u = q + 128 = 16 hi + lo, so sum u x = 16 D_hi + D_lo - 2176 sum x
                    // and sum q x = 16 D_hi + D_lo - 2304 sum x (the offset folds in below)
                    if constexpr (FMT == UQ_INT8_SYM) d[e] = fmaf(16.0f, dd[1][e], dd[0][e]);
                    else d[e] = dd[0][e] + dd[1][e];
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if constexpr (FMT == UQ_K4) {
                        float dsc, dmm;
                        row_meta_k4(sm, g + 8 * j, gg, dsc, dmm);
                        const float off = fmaf(128.0f, dsc, dmm);
                        p[2 * j] = fmaf(dsc, d[2 * j], fmaf(-off, sxv.x, p[2 * j]));
                        p[2 * j + 1] = fmaf(dsc, d[2 * j + 1], fmaf(-off, sxv.y, p[2 * j + 1]));
                    } else {
                        float sc, zc;
                        row_meta<FMT>(rp[j], gg, sc, zc);
                        if constexpr (FMT == UQ_INT8_SYM) zc = 2304.0f;
                        const float szc = sc * zc;
                        p[2 * j] = fmaf(sc, d[2 * j], fmaf(-szc, sxv.x, p[2 * j]));
                        p[2 * j + 1] = fmaf(sc, d[2 * j + 1], fmaf(-szc, sxv.y, p[2 * j + 1]));
                    }
                }
            };
            // one group, folded into p (p = acc for A8; a pair's sum from zero otherwise)
            auto group_step = [&](const int gg, float (&p)[4]) {
                if constexpr (A8) {
                    group_a8(gg, p);
                } else {
                    float dd[2][4];
                    group_mma(gg, dd, true, false);
                    fold(gg, dd, p);
                }
            };
            if constexpr (A8) {
                if (ng == GPT) {
                    constexpr int GUNROLL = (GB == 2) ? 8 : 4;
#pragma unroll GUNROLL
                    for (int gg = 0; gg < GPT; ++gg) group_step(gg, acc);
                } else {
#pragma unroll 1
                    for (int gg = 0; gg < ng; ++gg) group_step(gg, acc);
                }
            } else {
                // The tile's sum in rounds of 8 groups (the order gemv_warp_kernel's columns give):
                // each pair of groups folded from zero, p_q for groups 8r + 2q, 8r + 2q + 1, then
                // acc += (p_0 + p_1) + (p_2 + p_3).  `full`: a whole tile, whose groups all lie inside K.
                auto pair_step = [&](const int r, const int q, const bool full, float (&p)[4]) {
                    p[0] = p[1] = p[2] = p[3] = 0.f;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int gg = 8 * r + 2 * q + h;
                        if (full ? (GPT >= 8 || 2 * q + h < GPT) : gg < ng) group_step(gg, p);
                    }
                };
                auto round_step = [&](const int r, const bool full) {
                    float s01[4], sh[4], p[4];
                    // halves of the round (pairs 0, 1 then 2, 3): 4 groups per iteration (8 for
                    // 32-k groups), as deep as the compute warps' registers allow
                    constexpr int HUNROLL = (GB == 2) ? 2 : 1;
#pragma unroll HUNROLL
                    for (int hf = 0; hf < 2; ++hf) {
                        pair_step(r, 2 * hf, full, sh);
                        pair_step(r, 2 * hf + 1, full, p);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            sh[e] += p[e];
                            if (hf == 0) s01[e] = sh[e];
                            else acc[e] += s01[e] + sh[e];
                        }
                    }
                };
                // One row of x: round r's groups in the mma's columns (chains over the whole round;
                // blocks of other groups add exact zeros to a column), then lane (g, c) folds groups
                // 8r + 2c, 8r + 2c + 1 of rows g, g + 8 from zero and two shuffles add the four lanes'
                // pairs: the same operations on the same values as round_step, in the same order.
                auto round_col = [&](const int r, const bool full) {
                    float dd[2][4];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int gg = 8 * r + q;
                        if (full ? (GPT >= 8 || q < GPT) : gg < ng) group_mma(gg, dd, q == 0, true);
                    }
                    float d[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if constexpr (FMT == UQ_INT8_SYM) d[e] = fmaf(16.0f, dd[1][e], dd[0][e]);
                        else d[e] = dd[0][e] + dd[1][e];
                    }
                    float p[2] = {0.f, 0.f};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int gg = 8 * r + 2 * c + e;
                        if (!(full ? (GPT >= 8 || 2 * c + e < GPT) : gg < ng)) continue;
                        const float sx = sxc[gg * 8];
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            if constexpr (FMT == UQ_K4) {
                                float dsc, dmm;
                                row_meta_k4(sm, g + 8 * j, gg, dsc, dmm);
                                const float off = fmaf(128.0f, dsc, dmm);
                                p[j] = fmaf(dsc, d[2 * j + e], fmaf(-off, sx, p[j]));
                            } else {
                                float sc, zc;
                                row_meta<FMT>(rp[j], gg, sc, zc);
                                if constexpr (FMT == UQ_INT8_SYM) zc = 2304.0f;
                                const float szc = sc * zc;
                                p[j] = fmaf(sc, d[2 * j + e], fmaf(-szc, sx, p[j]));
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float s2 = p[j] + __shfl_xor_sync(0xffffffffu, p[j], 1);
                        acc[2 * j] += s2 + __shfl_xor_sync(0xffffffffu, s2, 2);
                    }
                };
                // (8 groups per round: a K4 record, 8 sub-blocks, is read and decoded once per row per
                // round, its 6-bit fields at constant shifts)
                if constexpr (COL) {
                    if (ng == GPT) {
#pragma unroll 1
                        for (int r = 0; r < (GPT + 7) / 8; ++r) round_col(r, true);
                    } else {
#pragma unroll 1
                        for (int r = 0; 8 * r < ng; ++r) round_col(r, false);
                    }
                } else if (ng == GPT) {
#pragma unroll 1
                    for (int r = 0; r < (GPT + 7) / 8; ++r) round_step(r, true);
                } else {
#pragma unroll 1
                    for (int r = 0; 8 * r < ng; ++r) round_step(r, false);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);                   // this warp's half of the slot is free
        slot += PWn;
        if (slot >= S2) { slot -= S2; ph ^= 1u; }
        if (kb < a.KB) {
            // the tile's partial sums: shared memory (cta_rows; slot = the tile's index in the CTA's
            // range) or global memory (slot = the tile's index in k-major order), summed over k later
            // (A8: scaled by the columns' s_x)
            if (cta_rows) {
                float* part = cpart + (2 * pl + hh) * RB * 8;
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) part[(g + 8 * j) * 8 + 2 * c + e] = A8 ? acc[2 * j + e] * sxm[e] : acc[2 * j + e];
            } else {
                float* part = a.partials + ((long long)kb * a.NB + nbw) * RB * M;
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (2 * c + e < M) part[(g + 8 * j) * M + 2 * c + e] = A8 ? acc[2 * j + e] * sxm[e] : acc[2 * j + e];
            }
        }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    }
    if (!cta_rows) return;
    // cta_rows: each row's sum over the k tiles, in k order, once every compute warp's tiles are in
    compute_warps_sync();
    auto row_sum = [&](int rbi, int r, int m) {         // tile (kb, rbi) is local tile 2 ((kb / 2) R + rbi) + kb % 2
        float sum = 0.f;
        for (int kb = 0; kb < L.KB; ++kb) sum += cpart[((2 * ((kb >> 1) * R + rbi) + (kb & 1)) * RB + r) * 8 + m];
        return sum;
    };
    for (int e = threadIdx.x; e < (R / WU) * RB * M; e += CW * 32) {
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

// ------------------------------------------------------------------------------------------------
// One row of x (M = 1) on the 4-bit formats: gemv_warp_kernel, the same per-tile arithmetic on
// per-warp rings.  Each warp owns its tiles and a ring of two stages (one computed, one in flight),
// copied by its own lanes with 16-byte cp.async in one cp.async group per tile, and a double-
// buffered slice of x (one bulk copy per k tile run).  Two CTAs of 4 warps per SM: each CTA's
// shared memory (~105 KB) leaves room for a CTA of the next kernel on the stream, which with launch
// overlap starts streaming its weights while this kernel's last CTAs finish.  A decode step's
// launches at M = 1 are short (~10 us for 30 MB), so that overlap of consecutive launches is worth
// more there than gemv_warp_kernel's deeper shared ring, which needs the whole SM.
//
// Tile order is k-major: tile i of a range is (k tile i / R, row block i % R) for R row blocks, so
// a warp's consecutive tiles share their k tile; the sums of x over the k tile's groups are formed
// once per run of equal k tile, in the order gemv_warp_kernel's table uses.  Every tile's partial
// sums are stored (shared memory when the CTA owns whole row blocks, global memory otherwise) and
// summed over the k tiles in k order afterwards, as gemv_warp_kernel does.
template <int FMT> struct WarpCfg {
    static constexpr int WARPS = 4;                                // workers per CTA
    static constexpr int STAGES = 2;                               // tiles in flight per worker
};
constexpr int WARP_CTAS_PER_SM = 2;
constexpr int WARP_TPW = 6;        // tiles per warp at most when the CTA owns whole row blocks

// bytes per row of an x slice (KT k of each row; 32 bytes of padding when there are two rows put
// the rows a half-warp's 8-byte B-fragment loads touch into different banks)
__host__ __device__ inline int gemv_warp_xslice_stride(int fmt, int M) {
    return M <= 1 ? fmt_kt(fmt) * 2 : fmt_kt(fmt) * 2 + 32;
}

// Shared memory: rings [warps][stages][stage] | ring and x-slice mbarriers | sums of x [warps][groups
// of a tile][8] | partial sums [tiles of the CTA, at most warps x WARP_TPW][16][8] | x slices
// [warps][2][M] | zeros [warps][320 bytes: 256 from byte 32] (the B fragments of the other groups'
// columns; 32 bytes off the x slices' alignment, so a load's x and zero lanes hit different banks)
__host__ __device__ inline GemvSmem gemv_warp_smem(int fmt, int group, int M) {
    int stage = 0, warps = 0;
    const int kt = fmt_kt(fmt);
    switch (fmt) {
        case UQ_INT4_SYM: stage = MetaGeom<UQ_INT4_SYM>::STAGE_BYTES; warps = WarpCfg<UQ_INT4_SYM>::WARPS; break;
        default: stage = MetaGeom<UQ_INT4_ASYM>::STAGE_BYTES; warps = WarpCfg<UQ_INT4_ASYM>::WARPS; break;
    }
    const int stages = 2;
    GemvSmem p;
    p.bars = (size_t)warps * stages * stage;
    p.lut = p.bars + (size_t)(warps * stages + 2 * warps) * 8;      // ring and x-slice mbarriers
    p.sx = (p.lut + 15) / 16 * 16;
    p.ps = p.sx + (size_t)warps * (kt / group) * 8 * 4;
    p.x = (p.ps + (size_t)warps * WARP_TPW * RB * 8 * 4 + 127) / 128 * 128;
    p.zr = p.x + (size_t)warps * 2 * M * gemv_warp_xslice_stride(fmt, M);
    p.total = p.zr + (size_t)warps * 320;
    return p;
}
// within the shared memory that keeps WARP_CTAS_PER_SM CTAs on an SM
constexpr int WARP_SMEM_LIMIT = (228 * 1024) / WARP_CTAS_PER_SM - 1024;
// the launches gemv_warp_kernel takes: one row of x on the 4-bit flat formats (measured faster there
// than gemv_mma_kernel; the 2-bit formats, K4 and more rows have more work per byte, where
// gemv_mma_kernel's 12 compute warps per SM are faster)
__host__ __device__ inline bool gemv_warp_route(int fmt, int M) {
    return M == 1 && (fmt == UQ_INT4_SYM || fmt == UQ_INT4_ASYM);
}

// GATED: the gated projection in one launch.  The work list interleaves the gate and up weights' row
// blocks (work row block 2j = gate row block j, 2j + 1 = up row block j), every CTA owns whole pairs,
// and the per-row reduction forms h = silu(g) * u (or the second pass does, for the stream-K split).
template <int FMT, int GB, bool GATED>
__global__ void __launch_bounds__(WarpCfg<FMT>::WARPS * 32, WARP_CTAS_PER_SM) gemv_warp_kernel(const GemvArgs a) {
    using F = GemvFmt<FMT>;
    static_assert(FMT == UQ_INT4_SYM || FMT == UQ_INT4_ASYM, "one row of x on the 4-bit flat formats");
    constexpr int KT = F::KT, S = WarpCfg<FMT>::STAGES, W = WarpCfg<FMT>::WARPS;
    constexpr int GS = GB * 16;                                     // k per scaling group
    constexpr int GPT = KT / GS;                                    // groups per full tile row (8, 16, 32)
    static_assert(GPT % 8 == 0, "rounds of 8 groups");
    constexpr int WPG = GB;                                         // code words per lane per group
    constexpr int BPCH = F::BPC;                                    // 16-k blocks per 512-byte chunk
    extern __shared__ __align__(128) uint8_t smem[];
    const int M = a.M;
    if (M != 1) {                                                   // the host routes one row of x here only
        if (threadIdx.x == 0) atomicOr(a.fault, FAULT_GEMV_SPLIT);
        return;
    }
    const GemvSmem plan = gemv_warp_smem(FMT, a.group, M);
    const int XB = gemv_warp_xslice_stride(FMT, M);                 // x slice: bytes per row
    uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + plan.bars);
    uint8_t* xs = smem + plan.x;
    float* cpart = reinterpret_cast<float*>(smem + plan.ps);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const Layout L(a.N, a.K, FMT);
    uint8_t* ring = smem + (size_t)warp * S * MetaGeom<FMT>::STAGE_BYTES;
    uint64_t* bars = bars_all + warp * S;
    uint64_t* xsl_bar = bars_all + W * S + 2 * warp;               // this warp's two x-slice buffers
    float* sxw = reinterpret_cast<float*>(smem + plan.sx) + warp * GPT * 8;   // sums of x of the run's k tile
    uint8_t* xsl = xs + (size_t)warp * 2 * M * XB;                  // this warp's x-slice buffers
    uint8_t* zrw = smem + plan.zr + warp * 320 + 32;                // this warp's 256 bytes of zeros
    const uint8_t* xz = zrw + 8 * c;

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
    if (cta_rows && ntl > WARP_TPW) {                                // the host never splits this way
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
    reinterpret_cast<uint32_t*>(zrw)[lane] = 0u;
    reinterpret_cast<uint32_t*>(zrw)[lane + 32] = 0u;
    __syncwarp();
    int issued = 0;                                                 // tiles requested so far
    // the weight and weight row block of a work row block
    const GemvSrc src_gate{a.wq, a.scales, a.zc}, src_up{a.wq2, a.scales2, a.zc2};
    // k-major tile coordinates (k tile, row block index in [0, R)) are advanced incrementally: a
    // 64-bit division per tile would cost more than the tile's scale folds
    int ikb = ntl > 0 ? kb_of(t0) : 0, irb = ntl > 0 ? (int)(t0 % R) : 0;   // the next tile to request
    auto issue_next = [&]() {
        const int nbw = rb0 + irb;
        issue_tile<FMT, GPT>(a, (GATED && (nbw & 1)) ? src_up : src_gate, L, mc, GATED ? nbw >> 1 : nbw, ikb,
                             ring + (issued % S) * MetaGeom<FMT>::STAGE_BYTES, lane);
        if (++irb == R) { irb = 0; ++ikb; }
        ++issued;
    };
    // Only the first tile before the sums of x of the first run: at the start every warp of the
    // GPU requests its tiles at once and a copy's issue waits for room in the memory system, so
    // the second tile is requested once this warp's sums of x are done (the memory system is
    // still busy with the first tiles then).
    if (a.overlap && has_work && ntl > 0) issue_next();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (has_work && ntl > 0 && lane == 0) {
        issue_xslice(kb_first, 0);
        if (kb_last > kb_first) issue_xslice(kb_first + 1, 1);
    }
    int xissued = (ntl > 0) ? ((kb_last > kb_first) ? 2 : 1) : 0;   // x-slice runs requested so far
    if (has_work && issued == 0 && ntl > 0) issue_next();
    if (!has_work) return;                          // (never in cta_rows mode: every warp meets the end barrier)

    int cur_kb = -1, run = -1;
    const uint8_t* xt = nullptr;                 // this lane's x at the current k tile's first k

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
            {
                const int slot = run & 1;
                bool ok = mbar_wait_bounded(&xsl_bar[slot], (uint32_t)((run >> 1) & 1), a.fault, FAULT_GEMV_WAIT);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (run >= 1 && kb + 1 <= kb_last) {
                    __syncwarp();                                   // the buffer's previous run is done
                    if (lane == 0) issue_xslice(kb + 1, slot ^ 1);
                    ++xissued;
                }
                xt = xsl + slot * XB + 8 * c;                       // (one row of x)
            }
            __syncwarp();                                           // the previous run's sums are read
            {
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
            }
            __syncwarp();
        }
        while (issued < ntl && issued < li + S) issue_next();        // top up the ring (into stages consumed)
        const int s = li % S;
        uint8_t* st = ring + s * MetaGeom<FMT>::STAGE_BYTES;
        // this tile's copies (one cp.async group) are complete once at most the groups of later
        // tiles are pending
        static_assert(S == 2, "one later group at most");
        if (issued > li + 1) cp_async_wait_group<1>();
        else cp_async_wait_group<0>();
        __syncwarp();
        RowPtrs<FMT> rp[2];
        rp[0] = row_ptrs<FMT>(st, mc, g, n0 + g, kb);
        rp[1] = row_ptrs<FMT>(st, mc, g + 8, n0 + g + 8, kb);

        // Round r: groups 8r .. 8r + 7 of the tile, one per column of the mma.  Lane group g feeds x
        // of group 8r + g as its B column and zeros for the other groups' blocks, so column i of D
        // is the sum over group 8r + i of (128 + q) x; blocks of other groups add exact zeros to it,
        // and two chains (even / odd blocks) sum it as gemv_mma_kernel does per group.  Lane (g, c)
        // folds groups 8r + 2c and 8r + 2c + 1 of rows g, g + 8 from zero, and two shuffles add the
        // four lanes' pairs: acc += (p_0 + p_1) + (p_2 + p_3), gemv_mma_kernel's order, so a row's
        // result is the same as in a batch.  The scales and zero points are read once per group and
        // row instead of once per group, row and lane.  `full`: a whole tile (all groups inside K).
        float acc[2] = {0.f, 0.f};                  // rows g, g + 8 (the one column of y)
        auto round_step = [&](const int r, const bool full) {
            float dd[2][4];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int gg = 8 * r + q;
                if (!full && gg >= ng) continue;
                // this lane's code words for the group's GB blocks
                uint32_t wv[GB];
                const int blk = gg * GB;                            // first block of the group in the tile
                const uint8_t* cp = st + (blk / BPCH) * CHUNK + lane * 16 + ((blk % BPCH) * WPG / GB) * 4;
                if constexpr (GB == 8) {
                    const uint4 v0 = *reinterpret_cast<const uint4*>(cp);
                    const uint4 v1 = *reinterpret_cast<const uint4*>(cp + CHUNK);
                    wv[0] = v0.x; wv[1] = v0.y; wv[2] = v0.z; wv[3] = v0.w;
                    wv[4] = v1.x; wv[5] = v1.y; wv[6] = v1.z; wv[7] = v1.w;
                } else if constexpr (GB == 4) {
                    const uint4 v = *reinterpret_cast<const uint4*>(cp);
                    wv[0] = v.x; wv[1] = v.y; wv[2] = v.z; wv[3] = v.w;
                } else {
                    const uint2 v = *reinterpret_cast<const uint2*>(cp);
                    wv[0] = v.x; wv[1] = v.y;
                }
                // B fragments: x at k = 16 blk + 4c .. +3 for the group's own column, else zeros
                const uint8_t* xb = (g == q) ? xt + blk * 32 : xz;
#pragma unroll
                for (int j = 0; j < GB; ++j) {
                    const uint2 v = *reinterpret_cast<const uint2*>(xb + j * 32);
                    const uint32_t wd = wv[j];
                    const uint32_t a0 = nib_pair_lop3<0>(wd), a1 = nib_pair_lop3<1>(wd);
                    const uint32_t a2 = nib_pair_lop3<2>(wd), a3 = nib_pair_lop3<3>(wd);
                    if (q == 0 && j < 2) mma_bf16_zero(dd[j & 1], a0, a1, a2, a3, v.x, v.y);
                    else mma_bf16(dd[j & 1], a0, a1, a2, a3, v.x, v.y);
                }
            }
            // lane (g, c) holds rows g, g + 8 of columns 2c, 2c + 1: groups 8r + 2c, 8r + 2c + 1
            float d[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) d[e] = dd[0][e] + dd[1][e];
            float p[2] = {0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int gg = 8 * r + 2 * c + e;
                if (!full && gg >= ng) continue;
                const float sx = sxw[gg * 8];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float sc, zc;
                    row_meta<FMT>(rp[j], gg, sc, zc);
                    const float szc = sc * zc;
                    p[j] = fmaf(sc, d[2 * j + e], fmaf(-szc, sx, p[j]));
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float s2 = p[j] + __shfl_xor_sync(0xffffffffu, p[j], 1);
                acc[j] += s2 + __shfl_xor_sync(0xffffffffu, s2, 2);
            }
        };
        if (ng == GPT) {
#pragma unroll
            for (int r = 0; r < GPT / 8; ++r) round_step(r, true);
        } else {
#pragma unroll 1
            for (int r = 0; 8 * r < ng; ++r) round_step(r, false);
        }
        __syncwarp();

        // the tile's partial sums (every lane holds them; lanes c = 0 store): shared memory
        // (cta_rows) or global memory, summed over k tiles later
        if (c == 0) {
            if (cta_rows) {
                float* part = cpart + (i * RB) * 8;                 // slot = the tile's index in the CTA's range
                part[g * 8] = acc[0];
                part[(g + 8) * 8] = acc[1];
            } else {
                float* part = a.partials + i * RB;                  // (one row of x)
                part[g] = acc[0];
                part[g + 8] = acc[1];
            }
        }
    }
    // a wait that timed out (fault flag set) left copies in flight: let them land before leaving
    cp_async_wait_group<0>();
    for (int r = (run > 0 ? run : 0); r < xissued; ++r)
        mbar_wait_bounded(&xsl_bar[r & 1], (uint32_t)((r >> 1) & 1), a.fault, FAULT_GEMV_WAIT);
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


namespace gemv_detail {
template <int FMT, int GB, int XM, bool GATED, bool A8 = false>
cudaError_t launch_mma(const GemvArgs& a, int grid, int sxg, cudaStream_t st) {
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gemv_mma_kernel<FMT, GB, XM, GATED, A8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 MMA_SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int threads = (MMA_CW + 1) * 32;
    GemvArgs a2 = a;
    a2.overlap = launch_overlap() ? 1 : 0;
    const MmaSmem plan = gemv_mma_smem(FMT, a.K, a.group, a.M, sxg, a.cta_rows, XM, A8 ? 1 : 2);
    a2.ring_slots = plan.S2;
    a2.sx_groups = sxg;
    a2.mma_pairs = gemv_mma_pairs(FMT, A8);
    if (a2.overlap) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = plan.total;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, gemv_mma_kernel<FMT, GB, XM, GATED, A8>, a2);
        if (e != cudaSuccess) return e;
    } else {
        gemv_mma_kernel<FMT, GB, XM, GATED, A8><<<grid, threads, plan.total, st>>>(a2);
    }
    return cudaGetLastError();
}
template <int FMT, int GB, bool GATED, bool A8 = false>
cudaError_t launch_mma_x(const GemvArgs& a, int grid, cudaStream_t st) {
    const int sxg = gemv_mma_sx_groups(FMT, a.group, a.NB, a.KB, grid, a.cta_rows);
    const int xm = gemv_mma_xmode(FMT, a.K, a.group, a.M, sxg, a.cta_rows, A8 ? 1 : 2, !A8 && !GATED);
    if constexpr (!A8 && !GATED)
        if (xm == MMA_X_ROW1) return launch_mma<FMT, GB, MMA_X_ROW1, GATED, A8>(a, grid, sxg, st);
    if (xm == MMA_X_WHOLE) return launch_mma<FMT, GB, MMA_X_WHOLE, GATED, A8>(a, grid, sxg, st);
    return launch_mma<FMT, GB, MMA_X_GLOBAL, GATED, A8>(a, grid, sxg, st);
}
template <int FMT, int GB, bool GATED>
cudaError_t launch_warp(const GemvArgs& a, int grid, cudaStream_t st) {
    static bool configured[64] = {};
    const size_t smem = gemv_warp_smem(FMT, a.group, a.M).total;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gemv_warp_kernel<FMT, GB, GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 WARP_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int threads = WarpCfg<FMT>::WARPS * 32;
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
        e = cudaLaunchKernelEx(&cfg, gemv_warp_kernel<FMT, GB, GATED>, a2);
        if (e != cudaSuccess) return e;
    } else {
        gemv_warp_kernel<FMT, GB, GATED><<<grid, threads, smem, st>>>(a2);
    }
    return cudaGetLastError();
}
template <int FMT, int GB, bool GATED>
cudaError_t launch_mma_xg(const GemvArgs& a, int grid, cudaStream_t st) {
    if constexpr (FMT == UQ_INT4_SYM || FMT == UQ_INT4_ASYM)
        if (gemv_warp_route(FMT, a.M)) return launch_warp<FMT, GB, GATED>(a, grid, st);
    return launch_mma_x<FMT, GB, GATED>(a, grid, st);
}
template <int FMT, int GB>
cudaError_t launch_mma_xs(const GemvArgs& a, int grid, cudaStream_t st) {
    return a.gated ? launch_mma_xg<FMT, GB, true>(a, grid, st) : launch_mma_xg<FMT, GB, false>(a, grid, st);
}
}  // namespace gemv_detail

template <int FMT>
cudaError_t launch_gemv_fmt(const GemvArgs& a, int grid, cudaStream_t st) {
    const int gs = (FMT == UQ_K4) ? 32 : a.group;
    switch (gs) {
        case 32: return gemv_detail::launch_mma_xs<FMT, 2>(a, grid, st);
        case 64: if constexpr (FMT != UQ_K4) return gemv_detail::launch_mma_xs<FMT, 4>(a, grid, st);
                 return cudaErrorInvalidValue;
        case 128: if constexpr (FMT != UQ_K4) return gemv_detail::launch_mma_xs<FMT, 8>(a, grid, st);
                  return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace uq
