// uq_tc.cu -- tensor-core fused dequantize + GEMM for M >= 16 (tcgen05, sm_103a).
//
// "Ultra LLM Engine", section "Fused Kernels": the dequantized-weight GEMM of batched decode.
// With 16..64 activation rows the product is a dense contraction, so it runs on the 5th-gen
// tensor cores; the kernel still streams each packed weight byte from HBM exactly once.
//
// Operands (swap-AB: the 128 weight rows are the MMA's M dimension, the activation rows its N):
//   A  = the integer part of the weights, (q - z) for INT4/INT8 and q for K4, exact in bf16,
//        written by the dequant warpgroup straight into TENSOR MEMORY (tcgen05.st), so the
//        dequantized operand never crosses shared memory;
//   B  = x, a [Mpad x 64] bf16 tile per 64-k step, loaded by TMA with the 128-byte swizzle
//        (the canonical K-major layout the MMA reads through a shared-memory descriptor);
//   D  = one fp32 accumulator slot in tensor memory per quantization group (128 lanes x Mpad
//        columns); the epilogue warpgroup reads it back (tcgen05.ld) and applies the group's
//        scale in fp32: y += s_g * sum_k (q - z) x  (K4: d*sc_j * sum q x - dmin*m_j * sum x).
// So the products and the per-group sums are exact up to fp32 accumulation, as in the GEMV.
//
// Roles (512 threads, one CTA per SM, persistent over an equal contiguous range of units):
//   warp 0       producer: per unit kc/64 TMA boxes of x, counted on full[stage];
//   warps 1, 2   MMA issuers (one thread each; for Mpad <= 32 two of them, on alternate units):
//                per group g/16 tcgen05.mma (M=128, N=Mpad, K=16) into the issuer's slots;
//   warps 4..11  dequant: warp = one 16-row block; it copies its 2 KB of codes per unit itself
//                (cp.async, two units ahead), and lane (g, c) turns its fragment-order words
//                into (q - z) bf16 pairs and stores them with tcgen05.st.16x256b (the store
//                shape whose thread layout is the mma fragment's), kc/2 columns per unit;
//   warps 12..15 epilogue: thread = weight row; scales, accumulates over the row block's units,
//                then stores y, or a partial sum plus a ticket (the last contributor reduces
//                the partials in CTA order, so results are deterministic and nobody waits).
// Unit = (128-row block, chunk of 128 code bytes per row = kc codes).  Every wait is bounded
// (mbar_wait_bounded); on a timeout the roles stop, the CTA frees its tensor memory and leaves.
#include <cuda.h>

#include "uq_kernels.h"

namespace uq {

namespace {

constexpr int TC_THREADS = 512;
constexpr int TC_ROWS = 128;
constexpr int TC_STAGE_CODES = TC_ROWS * 128;     // bytes of codes per stage
constexpr int TMEM_COLS = 512;
constexpr int TC_BAR_BYTES = 2048;                 // barriers and flags after the stages
constexpr int TC_MAX_STAGES = 6;

__device__ __forceinline__ long long trange_begin(int c, long long U, int P) { return (long long)c * U / P; }
__device__ __forceinline__ int tworker_of(long long u, long long U, int P) {
    return (int)(((u + 1) * (long long)P - 1) / U);
}

// ---- tcgen05 / TMA wrappers ------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// 16 lanes x 256 bits per repetition, fragment layout of an m16n8 accumulator: thread t holds
// (lane t/4, columns 2(t%4), 2(t%4)+1) and (lane t/4 + 8, same columns); .x4 repeats it over 32 columns
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                 :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                    "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
                    "r"(v[14]), "r"(v[15]) : "memory");
}
__device__ __forceinline__ void tmem_st_16x256b_x2(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.16x256b.x2.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                    "r"(v[7]) : "memory");
}
__device__ __forceinline__ void tc_cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void tc_cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }
// Copy the aligned 32-bit words that cover bytes [lo, lo + len) of `base` into dst[0 .. nw) (word 0
// holds byte lo & ~3).  Words that would reach past `end` (the array's size) are assembled from byte
// loads instead, so nothing outside the array is read.
__device__ __forceinline__ void stage_span(uint32_t* dst, const uint8_t* base, long long lo, int len, long long end) {
    const long long w0 = lo & ~3ll;
    for (long long src = w0; src < lo + len; src += 4, ++dst) {
        if (src + 4 <= end) {
            tc_cp_async4(dst, base + src);
        } else {
            uint32_t v = 0;
            for (int b = 0; b < 4; ++b)
                if (src + b < end) v |= (uint32_t)__ldg(base + src + b) << (8 * b);
            *dst = v;
        }
    }
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(smem_u32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar)) : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row core groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(const void* p) {
    const uint64_t addr = smem_u32(p);
    return ((addr & 0x3FFFFull) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M = 128, N = mpad.
__host__ __device__ constexpr uint32_t idesc_bf16(int mpad) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(mpad >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

template <int FMT> struct TcFmt {
    static constexpr int KC = (FMT == UQ_INT8_SYM) ? 128 : 256;   // codes per row per unit
    static constexpr int ACOLS = KC / 2;                           // tensor-memory columns of A per unit
    // per-thread metadata rings (3 units deep): epilogue scale words per row, dequant zero words
    static constexpr int SWORDS = (FMT == UQ_K4) ? 4 : 5;
    static constexpr int EPI_RING = 3 * 128 * SWORDS * 4;           // bytes
    static constexpr int DQ_RING = (FMT == UQ_INT4_ASYM) ? 3 * 8 * 16 * 2 * 4 : 0;
};
constexpr int TC_DQ_WARPS = 8;                     // dequant warps (one 16-row block each)

}  // namespace

struct TcSmem {
    // barriers live after the stage buffers; offsets computed on the host and device alike
    static __host__ __device__ constexpr int x_bytes(int kc, int mpad) { return kc * mpad * 2; }
    static __host__ __device__ constexpr int stage_bytes(int kc, int mpad) {
        return TC_STAGE_CODES + x_bytes(kc, mpad);
    }
};

// GB = 16-k blocks per scaling group (2, 4 or 8); used by the INT4_ASYM zero points, ignored otherwise
template <int FMT, int MPAD, int GB>
__global__ void __launch_bounds__(TC_THREADS, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const TcArgs a) {
    constexpr int KC = TcFmt<FMT>::KC;
    constexpr int ACOLS = TcFmt<FMT>::ACOLS;
    constexpr int XB = TcSmem::x_bytes(KC, MPAD);
    constexpr int SB = TcSmem::stage_bytes(KC, MPAD);
    constexpr int SWORDS = TcFmt<FMT>::SWORDS;
    constexpr uint32_t IDESC = idesc_bf16(MPAD);
    constexpr int NISS = MPAD <= 32 ? 2 : 1;        // MMA issuing threads
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int S = a.stages, DS = a.dslots;
    const int G = (FMT == UQ_K4) ? 32 : a.group;   // scaling granularity (K4: the 32-weight sub-block)
    const int GPC = KC / G;                         // groups (K4: sub-blocks) per unit
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * SB);
    uint64_t* full = bars;                          // [S]
    uint64_t* empty = full + S;                     // [S]
    uint64_t* afull = empty + S;                    // [2]
    uint64_t* aempty = afull + 2;                   // [2]
    uint64_t* dfull = aempty + 2;                   // [DS]
    uint64_t* dempty = dfull + DS;                  // [DS]
    uint64_t* ebar = dempty + DS;                   // epilogue warpgroup rendezvous (128 arrivals)
    uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(ebar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_smem + 1);
    unsigned int* ticket_smem = reinterpret_cast<unsigned int*>(tmem_base_smem + 2);
    uint32_t* epi_ring = reinterpret_cast<uint32_t*>(smem + S * SB + TC_BAR_BYTES);          // [3][128][SWORDS]
    uint32_t* dq_ring = epi_ring + TcFmt<FMT>::EPI_RING / 4;                                // [3][8 warps][16][2]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = trange_begin(cta, a.U, a.P), u1 = trange_begin(cta + 1, a.U, a.P);

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&afull[i], TC_DQ_WARPS); mbar_init(&aempty[i], 1); }
        for (int d = 0; d < DS; ++d) { mbar_init(&dfull[d], 1); mbar_init(&dempty[d], 4); }
        mbar_init(ebar, 128);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0) tmem_alloc(tmem_base_smem, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_smem;
    const uint32_t A_COL0 = 0;                      // A buffers: columns [0, 2*ACOLS)
    const uint32_t D_COL0 = 2 * ACOLS;              // D slots: columns [2*ACOLS, 2*ACOLS + DS*MPAD)

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            int issued = 0;
            auto issue_x = [&](int c, int s) {
                uint8_t* st = smem + s * SB;
#pragma unroll
                for (int q = 0; q < KC / 64; ++q)
                    tma_load_2d(st + TC_STAGE_CODES + q * (MPAD * 128), &tmap_x, c * KC + q * 64, 0, &full[s]);
            };
            // x may be written by the kernel before on the stream: loaded after the wait for it (the
            // dequant warps request the codes themselves)
            const int pre = (u1 - u0) < S ? (int)(u1 - u0) : S;
            const int CH = a.CH;
            int rb = (int)(u0 / CH), c = (int)(u0 % CH);
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int j = 0; j < pre; ++j) {
                mbar_arrive_expect_tx(&full[j], (uint32_t)XB);
                issue_x(c, j);
                if (++c == CH) { c = 0; ++rb; }
            }
            issued = pre;
            int s = 0;
            uint32_t eph = 1;                                // empty[] of the first round counts as free
            for (long long u = u0 + pre; u < u1 && !*abort_flag; ++u, ++issued) {
                if (s == 0) eph ^= 1;
                if (!mbar_wait_bounded(&empty[s], eph, a.fault, FAULT_TC_WAIT)) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], (uint32_t)XB);
                issue_x(c, s);
                if (++c == CH) { c = 0; ++rb; }
                if (++s == S) s = 0;
            }
            // let the last copies land before the CTA can leave
            for (int j = issued - 1; j >= 0 && j >= issued - S; --j)
                mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1), a.fault, FAULT_TC_WAIT);
        }
    } else if (warp == 1 || (NISS == 2 && warp == 2)) {
        // ---------------------------------------------------------------- MMA issuers
        // A thread issuing tcgen05.mma is held for tens of cycles per instruction, longer than
        // MMAs with N <= 32 keep the tensor pipe busy, so there two threads issue: warp 1 the
        // CTA's even units (A buffer 0, accumulator slots [0, DH)), warp 2 the odd ones (A buffer
        // 1, slots [DH, 2 DH)).  Each thread's MMAs and commits stay in its own order.
        if (lane == 0) {
            const int me = warp - 1, DH = DS / NISS;
            int d = 0;
            uint32_t dph = 0;                            // phase of dempty[me * DH + d] (^1)
            const int KS = G / 16;                       // MMAs per group
            for (long long u = u0 + me; u < u1 && !*abort_flag; u += NISS) {
                const int i = (int)(u - u0);
                const int s = i % S, ab = i & 1;
                const uint32_t sph = (uint32_t)((i / S) & 1), aph = (uint32_t)((i >> 1) & 1);
                bool ok = mbar_wait_bounded(&full[s], sph, a.fault, FAULT_TC_WAIT) &&
                          mbar_wait_bounded(&afull[ab], aph, a.fault, FAULT_TC_WAIT);
                if (!ok) { *abort_flag = 1; break; }
                tc_fence_after();
                // B descriptors advance by 32 bytes per 16-k slice and by one x box (MPAD x 128 B)
                // per 64 k: the start-address field is byte address / 16
                const uint64_t bdesc0 = sw128_desc(smem + s * SB + TC_STAGE_CODES);
                const uint32_t acol0 = tmem + A_COL0 + ab * ACOLS;
                int ks = 0;
                for (int j = 0; j < GPC; ++j) {
                    const int slot = me * DH + d;
                    if (!mbar_wait_bounded(&dempty[slot], dph ^ 1u, a.fault, FAULT_TC_WAIT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dcol = tmem + D_COL0 + slot * MPAD;
                    for (int t = 0; t < KS; ++t, ++ks) {
                        const uint64_t bdesc = bdesc0 + (uint64_t)((ks >> 2) * (MPAD * 8) + (ks & 3) * 2);
                        mma_ts(dcol, acol0 + ks * 8, bdesc, IDESC, t > 0 ? 1u : 0u);
                    }
                    tc_commit(&dfull[slot]);
                    if (++d == DH) { d = 0; dph ^= 1u; }
                }
                if (!ok) { *abort_flag = 1; break; }
                tc_commit(&aempty[ab]);
                tc_commit(&empty[s]);
            }
        }
    } else if (warp >= 4 && warp < 4 + TC_DQ_WARPS) {
        // ---------------------------------------------------------------- dequant warps
        // warp -> one 16-row block of the unit, in the tensor-memory lane quarter (warp % 4) it may
        // access; lane (g, c) holds the fragment-order words of rows g and g + 8, which the 16x256b
        // store shape takes as they are: no shuffles, one 16-byte shared-memory read per 4 words.
        const int quarter = warp & 3, hf = (warp >= 8) ? 1 : 0;
        const int rbl = 2 * quarter + hf;               // row block (16 rows) within the 128-row unit
        const int g = lane >> 2, c4 = lane & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter + 16 * hf) << 16);
        uint32_t* zr = dq_ring + (warp - 4) * 32;       // this warp's slot: 16 rows x 2 words
        // Unit u's copies, two units ahead, one cp.async group per unit: this warp's 2 KB of codes
        // (16-row block rb * 8 + rbl, k tile c / 4, chunks (c % 4) * 4 .. + 3, contiguous in the
        // fragment-order plane) into stage (u - u0) % S, and for INT4_ASYM the zero-point words of
        // rows g and g + 8 (lanes c = 0, 1).  A single thread issuing the eight 2 KB bulk copies of
        // a unit could not keep up with the stream (~0.14 us per copy).
        auto issue_zeros = [&](long long u) {
            if (u < u1) {
                const int rbc = (int)u / a.CH, cc = (int)u % a.CH;
                if (rbc * 8 + rbl < a.NB) {
                    const uint8_t* src = a.wq + (long long)(rbc * 8 + rbl) * 16 * a.rowbytes + (long long)(cc >> 2) * 8192 +
                                         (cc & 3) * 4 * 512;
                    uint8_t* dst = smem + ((int)(u - u0) % S) * SB + rbl * 2048;
#pragma unroll
                    for (int q = 0; q < 4; ++q) tc_cp_async16(dst + q * 512 + lane * 16, src + q * 512 + lane * 16);
                }
            }
            if constexpr (FMT == UQ_INT4_ASYM) {
                if (u < u1 && c4 < 2) {
                    const int rb = (int)u / a.CH, c = (int)u % a.CH;
                    const int r = g + 8 * c4;
                    const long long n = (long long)rb * TC_ROWS + rbl * 16 + r;
                    const int Gn = a.K / G, ZB = (Gn + 1) >> 1;
                    if (n < a.N)
                        stage_span(zr + ((int)(u - u0) % 3) * (TC_DQ_WARPS * 32) + r * 2, a.zc,
                                   n * ZB + (long long)c * (GPC >> 1), GPC >> 1, (long long)a.N * ZB);
                }
            }
            cp_async_commit();
        };
        issue_zeros(u0);
        issue_zeros(u0 + 1);
        int s = 0, ab = 0, zslot = 0;
        uint32_t sph = 0, aph = 1;                      // full[s] phase; aempty[] of the first round is free
        int rb = (int)u0 / a.CH, c = (int)u0 % a.CH;
        for (long long u = u0; u < u1 && !*abort_flag; ++u) {
            __syncwarp();
            issue_zeros(u + 2);
            // subtrahend per group as a bf16 pair: 128 + z (INT4_ASYM), 128 + 8 (INT4_SYM), 128 (K4)
            constexpr int ZG = (FMT == UQ_INT4_ASYM) ? 16 / GB : 1;   // groups per unit
            uint32_t zlo[ZG], zhi[ZG];
#pragma unroll
            for (int j = 0; j < ZG; ++j) zlo[j] = zhi[j] = (FMT == UQ_INT4_SYM) ? 0x43084308u : 0x43004300u;
            cp_async_wait2();                               // unit u's codes (and zero words) landed
            __syncwarp();
            if constexpr (FMT == UQ_INT4_ASYM) {
                const int Gn = a.K / G, ZB = (Gn + 1) >> 1;
                const uint32_t* slot = zr + zslot * (TC_DQ_WARPS * 32);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const long long n = (long long)rb * TC_ROWS + rbl * 16 + g + 8 * h;
                    uint32_t zb = 0;
                    if (n < a.N) {
                        const int o = (int)((n * ZB + (long long)c * (GPC >> 1)) & 3);
                        const uint64_t w = (uint64_t)slot[(g + 8 * h) * 2] | ((uint64_t)slot[(g + 8 * h) * 2 + 1] << 32);
                        zb = (uint32_t)(w >> (8 * o));
                    }
#pragma unroll
                    for (int j = 0; j < ZG; ++j) {
                        const uint32_t z = (zb >> (4 * j)) & 15u;
                        const uint32_t zz = 0x43004300u | z | (z << 16);
                        if (h == 0) zlo[j] = zz; else zhi[j] = zz;
                    }
                }
            }
            bool ok = mbar_wait_bounded(&aempty[ab], aph, a.fault, FAULT_TC_WAIT);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) { *abort_flag = 1; break; }
            tc_fence_after();
            const uint8_t* rbase = smem + s * SB + rbl * 2048 + lane * 16;
            const uint32_t acol = lane_addr + A_COL0 + ab * ACOLS;
            if constexpr (FMT == UQ_INT8_SYM) {
                // chunk q = 32 k = blocks 2q, 2q + 1; word 2b + h = row g + 8h, k 4c .. 4c + 3 of block b
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(rbase + q * 512);
                    const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
                    uint32_t v[8];
#pragma unroll
                    for (int b = 0; b < 2; ++b)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t wd = wv[2 * b + h];
                            const float f0 = byte_magic_f32(wd, 0) - 8388736.0f;
                            const float f1 = byte_magic_f32(wd, 1) - 8388736.0f;
                            const float f2 = byte_magic_f32(wd, 2) - 8388736.0f;
                            const float f3 = byte_magic_f32(wd, 3) - 8388736.0f;
                            v[4 * b + 2 * h] = f32x2_to_bf16x2(f0, f1);
                            v[4 * b + 2 * h + 1] = f32x2_to_bf16x2(f2, f3);
                        }
                    tmem_st_16x256b_x2(acol + q * 16, v);
                }
            } else {
                // chunk q = 64 k = blocks 4q .. 4q + 3, one word each; pairs 0/2 are row g (k 4c, 4c+1 /
                // 4c+2, 4c+3), pairs 1/3 row g + 8
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(rbase + q * 512);
                    const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
                    uint32_t v[16];
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int j = (FMT == UQ_INT4_ASYM) ? (4 * q + b) / GB : 0;
                        v[4 * b + 0] = bf16x2_sub(nib_pair_lop3<0>(wv[b]), zlo[j]);
                        v[4 * b + 1] = bf16x2_sub(nib_pair_lop3<2>(wv[b]), zlo[j]);
                        v[4 * b + 2] = bf16x2_sub(nib_pair_lop3<1>(wv[b]), zhi[j]);
                        v[4 * b + 3] = bf16x2_sub(nib_pair_lop3<3>(wv[b]), zhi[j]);
                    }
                    tmem_st_16x256b_x4(acol + q * 32, v);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[ab]);
            if (++s == S) { s = 0; sph ^= 1u; }
            ab ^= 1;
            if (ab == 0) aph ^= 1u;
            if (++zslot == 3) zslot = 0;
            if (++c == a.CH) { c = 0; ++rb; }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // no copy lands after the CTA left
    } else if (warp >= 4 + TC_DQ_WARPS) {
        // ---------------------------------------------------------------- epilogue warpgroup
        asm volatile("griddepcontrol.wait;" ::: "memory");   // sx, workspace and y follow earlier work
        const int we = warp & 3;
        const int r = we * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(we * 32) << 16);
        uint32_t* er = epi_ring + r * SWORDS;            // this thread's slot (ring stride 128 * SWORDS)
        // this row's scale words (K4: its super-block record) staged three units ahead
        auto issue_scales = [&](long long u) {
            if (u < u1) {
                const int rb = (int)u / a.CH, c = (int)u % a.CH;
                const long long n = (long long)rb * TC_ROWS + r;
                uint32_t* dst = er + ((int)(u - u0) % 3) * (128 * SWORDS);
                if (n < a.N) {
                    if constexpr (FMT == UQ_K4) {
                        tc_cp_async16(dst, a.scales + (n * (a.K >> 8) + c) * 16);
                    } else {
                        const long long Gn = a.K / G;
                        stage_span(dst, a.scales, (n * Gn + (long long)c * GPC) * 2, GPC * 2, (long long)a.N * Gn * 2);
                    }
                }
            }
            cp_async_commit();
        };
        issue_scales(u0);
        issue_scales(u0 + 1);
        float acc[MPAD];
#pragma unroll
        for (int m = 0; m < MPAD; ++m) acc[m] = 0.f;
        // accumulator slots: unit u's groups are in the ring of the issuer that took it ((u - u0) mod
        // the issuer count), slots [DH * ring, DH * ring + DH), consumed in that issuer's order
        const int DH = DS / NISS;
        int dring[2] = {0, 0}, eslot = 0;
        uint32_t dphr[2] = {0u, 0u}, ephase = 0;
        // all 128 epilogue threads meet here (bounded: returns false after the time limit)
        auto epi_sync = [&]() -> bool {
            mbar_arrive(ebar);
            const bool r_ok = mbar_wait_bounded(ebar, ephase, a.fault, FAULT_TC_WAIT);
            ephase ^= 1u;
            return r_ok;
        };
        const int first_rb = (int)u0 / a.CH;
        int rb = first_rb, c = (int)u0 % a.CH;
        for (long long u = u0; u < u1 && !*abort_flag; ++u) {
            const int n = rb * TC_ROWS + r;
            const bool live = n < a.N;
            issue_scales(u + 2);
            cp_async_wait2();
            const uint32_t* sw = er + eslot * (128 * SWORDS);
            if (++eslot == 3) eslot = 0;
            const int so = live ? (int)(((long long)n * (a.K / G) + (long long)c * GPC) & 1) : 0;   // halves
            const int ring = NISS == 2 ? (int)((u - u0) & 1) : 0;
            int d = ring ? dring[1] : dring[0];
            uint32_t dph = ring ? dphr[1] : dphr[0];
            bool ok = true;
            for (int j = 0; j < GPC; ++j) {
                float s1 = 0.f, s2 = 0.f;
                if (live) {
                    if constexpr (FMT == UQ_K4) {
                        const uint4 rec = *reinterpret_cast<const uint4*>(sw);
                        const uint64_t sc48 = (uint64_t)rec.y | ((uint64_t)(rec.z & 0xFFFFu) << 32);
                        const uint64_t m48 = (uint64_t)(rec.z >> 16) | ((uint64_t)rec.w << 16);
                        s1 = half_bits_f32((uint16_t)(rec.x & 0xFFFF)) * (float)((sc48 >> (6 * j)) & 63);
                        s2 = half_bits_f32((uint16_t)(rec.x >> 16)) * (float)((m48 >> (6 * j)) & 63);
                    } else {
                        s1 = half_bits_f32(reinterpret_cast<const uint16_t*>(sw)[so + j]);
                    }
                }
                const int slot = ring * DH + d;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&dfull[slot], dph, a.fault, FAULT_TC_WAIT));
                if (!ok) break;
                tc_fence_after();
                // up to 32 columns per wait for the loads (more would spill beside acc[64])
                constexpr int QN = MPAD / 16, QB = QN < 2 ? QN : 2;
#pragma unroll
                for (int q0 = 0; q0 < QN; q0 += QB) {
                    float v[QB][16];
#pragma unroll
                    for (int q = 0; q < QB; ++q)
                        if (q0 + q < QN) tmem_ld16(lane_addr + D_COL0 + slot * MPAD + (q0 + q) * 16, v[q]);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < QB; ++q)
                        if (q0 + q < QN)
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                acc[(q0 + q) * 16 + e] = fmaf(s1, v[q][e], acc[(q0 + q) * 16 + e]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&dempty[slot]);
                if (++d == DH) { d = 0; dph ^= 1u; }
                if constexpr (FMT == UQ_K4) {
                    const float* sx = a.sx + (long long)((c * KC + j * 32) >> 5) * MPAD;
#pragma unroll
                    for (int m = 0; m < MPAD; ++m) acc[m] = fmaf(-s2, __ldg(sx + m), acc[m]);
                }
            }
            if (ring) { dring[1] = d; dphr[1] = dph; } else { dring[0] = d; dphr[0] = dph; }
            if (!ok) { *abort_flag = 1; break; }
            if (c == a.CH - 1 || u == u1 - 1) {
                // row block finished for this CTA: store y, or a partial and a ticket
                const bool fullcov = (c == a.CH - 1) && (rb != first_rb || (u0 % a.CH) == 0);
                if (fullcov) {
                    if (live)
#pragma unroll
                        for (int m = 0; m < MPAD; ++m)
                            if (m < a.M)
                                a.y[(long long)m * a.ldy + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[m]));
                } else {
                    const int slot = 2 * cta + (rb == first_rb ? 0 : 1);
                    float* part = a.partials + (long long)slot * TC_ROWS * MPAD + r;   // [slot][m][row]
#pragma unroll
                    for (int m = 0; m < MPAD; ++m) part[m * TC_ROWS] = acc[m];
                    __threadfence();
                    if (!epi_sync()) { *abort_flag = 1; break; }
                    if (r == 0) *ticket_smem = atomicAdd(a.tickets + rb, 1u);
                    if (!epi_sync()) { *abort_flag = 1; break; }
                    const unsigned int old = *ticket_smem;
                    const long long uf = (long long)rb * a.CH;
                    const int cf = tworker_of(uf, a.U, a.P), cl = tworker_of(uf + a.CH - 1, a.U, a.P);
                    if (old == (unsigned int)(cl - cf)) {
                        __threadfence();
                        // the partials of all contributors, summed in CTA order into acc
#pragma unroll
                        for (int m = 0; m < MPAD; ++m) acc[m] = 0.f;
                        for (int c2 = cf; c2 <= cl; ++c2) {
                            const int rb2 = (int)(trange_begin(c2, a.U, a.P) / a.CH);
                            const int slot2 = 2 * c2 + (rb == rb2 ? 0 : 1);
                            const float* p2 = a.partials + (long long)slot2 * TC_ROWS * MPAD + r;
#pragma unroll
                            for (int m = 0; m < MPAD; ++m) acc[m] += __ldcg(p2 + m * TC_ROWS);
                        }
                        if (live)
#pragma unroll
                            for (int m = 0; m < MPAD; ++m)
                                if (m < a.M)
                                    a.y[(long long)m * a.ldy + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[m]));
                        if (r == 0) a.tickets[rb] = 0u;
                    }
                    if (!epi_sync()) { *abort_flag = 1; break; }
                }
#pragma unroll
                for (int m = 0; m < MPAD; ++m) acc[m] = 0.f;
            }
            if (++c == a.CH) { c = 0; ++rb; }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
// column sums of x per 32-k block, for the K4 min term: sx[j][m] = sum_{k in block j} x[m][k]
__global__ void colsum32_kernel(const uint16_t* __restrict__ x, float* __restrict__ sx, int M, int mpad, int K,
                                int ldx) {
    const int J = K / 32;
    const long long total = (long long)J * mpad;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(i / mpad), m = (int)(i % mpad);
        float s0 = 0.f, s1 = 0.f;
        if (m < M) {
            const uint32_t* p = reinterpret_cast<const uint32_t*>(x + (long long)m * ldx + j * 32);
#pragma unroll
            for (int v = 0; v < 16; ++v) {
                const uint32_t w = p[v];
                const float t = bf16lo_f32(w) + bf16hi_f32(w);
                if (v < 8) s0 += t; else s1 += t;
            }
        }
        sx[i] = s0 + s1;
    }
}

// ---------------------------------------------------------------------------------------------
// host side

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

template <int FMT, int MPAD, int GB>
cudaError_t launch_tc_t(const CUtensorMap& mx, const TcArgs& a, size_t smem, int grid, cudaStream_t st) {
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(tc_kernel<FMT, MPAD, GB>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    if (launch_overlap()) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(TC_THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, tc_kernel<FMT, MPAD, GB>, mx, a);
        if (e != cudaSuccess) return e;
    } else {
        tc_kernel<FMT, MPAD, GB><<<grid, TC_THREADS, smem, st>>>(mx, a);
    }
    return cudaGetLastError();
}

template <int FMT, int GB>
cudaError_t launch_tc_mg(int mpad, const CUtensorMap& mx, const TcArgs& a, size_t smem, int grid,
                         cudaStream_t st) {
    switch (mpad) {
        case 16: return launch_tc_t<FMT, 16, GB>(mx, a, smem, grid, st);
        case 32: return launch_tc_t<FMT, 32, GB>(mx, a, smem, grid, st);
        case 48: return launch_tc_t<FMT, 48, GB>(mx, a, smem, grid, st);
        case 64: return launch_tc_t<FMT, 64, GB>(mx, a, smem, grid, st);
        default: return cudaErrorInvalidValue;
    }
}
template <int FMT>
cudaError_t launch_tc_m(int mpad, const CUtensorMap& mx, const TcArgs& a, size_t smem, int grid,
                        cudaStream_t st) {
    if constexpr (FMT == UQ_INT4_ASYM) {
        switch (a.group) {
            case 32: return launch_tc_mg<FMT, 2>(mpad, mx, a, smem, grid, st);
            case 64: return launch_tc_mg<FMT, 4>(mpad, mx, a, smem, grid, st);
            case 128: return launch_tc_mg<FMT, 8>(mpad, mx, a, smem, grid, st);
            default: return cudaErrorInvalidValue;
        }
    } else {
        return launch_tc_mg<FMT, 8>(mpad, mx, a, smem, grid, st);
    }
}
}  // namespace

bool tc_supported(int fmt, int N, int K) {
    if (fmt != UQ_INT4_SYM && fmt != UQ_INT4_ASYM && fmt != UQ_INT8_SYM && fmt != UQ_K4) return false;
    if (N < 1 || K % fmt_kt(fmt)) return false;
    return encode_fn() != nullptr;
}

int tc_plan(int fmt, int mpad, int* stages, int* dslots, size_t* smem) {
    const int kc = (fmt == UQ_INT8_SYM) ? 128 : 256;
    const int sb = TcSmem::stage_bytes(kc, mpad);
    int rings = 0;
    switch (fmt) {
        case UQ_INT4_SYM: rings = TcFmt<UQ_INT4_SYM>::EPI_RING + TcFmt<UQ_INT4_SYM>::DQ_RING; break;
        case UQ_INT4_ASYM: rings = TcFmt<UQ_INT4_ASYM>::EPI_RING + TcFmt<UQ_INT4_ASYM>::DQ_RING; break;
        case UQ_INT8_SYM: rings = TcFmt<UQ_INT8_SYM>::EPI_RING + TcFmt<UQ_INT8_SYM>::DQ_RING; break;
        case UQ_K4: rings = TcFmt<UQ_K4>::EPI_RING + TcFmt<UQ_K4>::DQ_RING; break;
        default: return -1;
    }
    const int budget = 227 * 1024 - 1024 - TC_BAR_BYTES - rings;
    int s = budget / sb;
    if (s > TC_MAX_STAGES) s = TC_MAX_STAGES;
    if (s < 3) return -1;                           // codes are requested two units ahead
    int ds = (TMEM_COLS - kc) / mpad;       // A takes 2 * kc/2 columns
    if (ds > 8) ds = 8;
    *stages = s;
    *dslots = ds;
    *smem = 1024 + (size_t)s * sb + TC_BAR_BYTES + rings;
    return 0;
}

cudaError_t launch_colsum32(const uint16_t* x, float* sx, int M, int mpad, int K, int ldx, cudaStream_t st) {
    const long long total = (long long)(K / 32) * mpad;
    int g = (int)((total + 255) / 256);
    if (g > 4096) g = 4096;
    colsum32_kernel<<<g < 1 ? 1 : g, 256, 0, st>>>(x, sx, M, mpad, K, ldx);
    return cudaGetLastError();
}

cudaError_t launch_tc(int fmt, const uint16_t* x, const TcArgs& a, size_t smem, int grid, cudaStream_t st) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap mx;
    {
        cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
        cuuint64_t strides[1] = {(cuuint64_t)a.ldx * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)a.Mpad};
        cuuint32_t es[2] = {1, 1};
        if (enc(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    switch (fmt) {
        case UQ_INT4_SYM: return launch_tc_m<UQ_INT4_SYM>(a.Mpad, mx, a, smem, grid, st);
        case UQ_INT4_ASYM: return launch_tc_m<UQ_INT4_ASYM>(a.Mpad, mx, a, smem, grid, st);
        case UQ_INT8_SYM: return launch_tc_m<UQ_INT8_SYM>(a.Mpad, mx, a, smem, grid, st);
        case UQ_K4: return launch_tc_m<UQ_K4>(a.Mpad, mx, a, smem, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace uq
