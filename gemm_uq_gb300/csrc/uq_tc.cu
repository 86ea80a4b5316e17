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

constexpr int TC_ROWS = 128;
constexpr int TMEM_COLS = 512;
constexpr int TC_BAR_BYTES = 2048;                 // barriers and flags after the stages

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
// D[tmem] (+)= A[tmem] * B[smem desc], executed by the whole (converged) warp: the operands are
// warp-uniform and the elected lane (the lowest active one) issues the instruction
__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// tcgen05.commit by the elected lane of the converged warp (the lane that issued the MMAs)
__device__ __forceinline__ void tc_commit_elect(uint64_t* bar) {
    asm volatile("{\n\t.reg .pred e;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
                 :: "r"(smem_u32(bar)) : "memory");
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
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
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

// cp.async.wait_group with a compile-time count
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

template <int FMT> struct TcFmt {
    static constexpr int BITS = fmt_bits(FMT);
    static constexpr int KC = (FMT == UQ_INT8_SYM || FMT == UQ_NF4) ? 128 : 256;   // codes per row per unit
    // A planes: NF4's non-integer codebook value c[q] is written as two bf16 planes, hi = bf16(c[q]) and
    // lo = bf16(c[q] - hi), multiplied into the same accumulator; the other formats' A is an exact integer
    static constexpr int PLANES = (FMT == UQ_NF4) ? 2 : 1;
    static constexpr int ACOLS = KC / 2 * PLANES;                  // tensor-memory columns of A per unit
    static constexpr int WBYTES = 16 * KC * BITS / 8;              // code bytes of one 16-row block per unit
    static constexpr int CODES = 8 * WBYTES;                       // code bytes per unit (128 rows)
    static constexpr int CPU = KC / fmt_kc(FMT);                   // 512-byte chunks per 16-row block per unit
    // staged scale words per row and unit: the unit's KC / (16 GB) fp16 scales plus one half for a
    // start that is not word aligned (K4: its 16-byte super-block record)
    template <int GB> static constexpr int swords() { return FMT == UQ_K4 ? 4 : (KC / (16 * GB) + 2) / 2; }
};
constexpr int TC_DQ_WARPS = 8;                     // dequant warps (one 16-row block each)
// Epilogue warps: one per tensor-memory lane quarter for Mpad <= 32 (all columns), two per quarter
// above (half the columns each, so the per-thread accumulators fit in registers)
__host__ __device__ constexpr int tc_epi_warps(int mpad) { return mpad >= 48 ? 8 : 4; }
__host__ __device__ constexpr int tc_threads(int mpad) { return (4 + TC_DQ_WARPS + tc_epi_warps(mpad)) * 32; }
constexpr int TC_EPI_RING = 8;                     // epilogue scale ring: units staged 7 ahead

}  // namespace

// Shared-memory plan of the tensor-core kernel, the same on host and device:
//   [x ring: XS stages of one unit's x tile][code ring: CS stages of one unit's 16 KB of codes]
//   [barriers][epilogue scale ring][INT4_ASYM zero-point ring]
// The code ring is separate from the x ring and deeper: the dequant warps request their codes
// CS - 1 units ahead, which keeps enough bytes in flight per SM to cover the memory latency.
template <int FMT, int MPAD, int GB> struct TcPlan {
    static constexpr int KC = TcFmt<FMT>::KC;
    static constexpr int XB = KC * MPAD * 2;                       // x bytes per unit (MPAD rows x KC k)
    static constexpr int XS = 4;                                   // x stages
    static constexpr int EPI_RING = TC_EPI_RING * 32 * tc_epi_warps(MPAD) * TcFmt<FMT>::template swords<GB>() * 4;
    // zero-point words staged per row and unit: INT4_ASYM two (its nibbles), INT2_ASYM the unit's fp16 zeros
    static constexpr int ZW = FMT == UQ_INT4_ASYM ? 2 : (FMT == UQ_INT2_ASYM ? (KC / (16 * GB) + 2) / 2 : 0);
    static constexpr int DQ_SLOT = TC_DQ_WARPS * 16 * ZW * 4;     // zero words per unit
    static constexpr int BUDGET = 227 * 1024 - 1024 - TC_BAR_BYTES - EPI_RING - XS * XB;
    static constexpr int CS_FIT = BUDGET / (TcFmt<FMT>::CODES + DQ_SLOT);
    static constexpr int CS = CS_FIT > 8 ? 8 : (CS_FIT > 4 && XB >= 24 * 1024 ? 4 : CS_FIT);   // code stages
    static constexpr int CD = CS - 1;                              // code prefetch depth (units)
    static constexpr int DS_FIT = (TMEM_COLS - 2 * TcFmt<FMT>::ACOLS) / MPAD;
    static constexpr int DS = DS_FIT > 8 ? 8 : DS_FIT;           // accumulator slots
    // A buffers: at least two, more where tensor memory has room beside the accumulator slots (the
    // dequant warps then run further ahead of the MMAs that free a buffer)
    static constexpr int NA_FIT = (TMEM_COLS - DS * MPAD) / TcFmt<FMT>::ACOLS;
    static constexpr int NA = NA_FIT > 4 ? 4 : NA_FIT;
    static_assert(NA >= 2, "two A buffers at least");
    static constexpr int CODE_OFF = XS * XB;
    static constexpr int BAR_OFF = CODE_OFF + CS * TcFmt<FMT>::CODES;
    static constexpr int EPI_OFF = BAR_OFF + TC_BAR_BYTES;
    static constexpr int DQ_OFF = EPI_OFF + EPI_RING;
    static constexpr int SMEM = 1024 + DQ_OFF + CS * DQ_SLOT;      // + alignment slack
    static_assert(CS >= 3, "the code ring needs at least three stages");
    static_assert(SMEM <= 227 * 1024, "shared memory plan too large");
};

// GB = 16-k blocks per scaling group (2, 4 or 8); used by the INT4_ASYM zero points, ignored otherwise
template <int FMT, int MPAD, int GB>
__global__ void __launch_bounds__(tc_threads(MPAD), 1)
tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const TcArgs a) {
    using PL = TcPlan<FMT, MPAD, GB>;
    constexpr int KC = TcFmt<FMT>::KC;
    constexpr int ACOLS = TcFmt<FMT>::ACOLS;
    constexpr int XB = PL::XB, XS = PL::XS, CS = PL::CS, CD = PL::CD, DS = PL::DS, NA = PL::NA;
    constexpr int SWORDS = TcFmt<FMT>::template swords<GB>();
    constexpr uint32_t IDESC = idesc_bf16(MPAD);
    // Two warps issue MMAs: for Mpad <= 32 on alternate units; for larger Mpad (4-bit codes) both on
    // every unit, each with half of its groups (SPLIT); INT8 at larger Mpad has one group per unit, one issuer
    constexpr bool SPLIT = MPAD >= 48 && KC == 256;
    constexpr int NISS = (MPAD <= 32 || SPLIT) ? 2 : 1;
    constexpr int EW = tc_epi_warps(MPAD);
    constexpr int HW = MPAD / (EW / 4);             // columns per epilogue warp
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int G = (FMT == UQ_K4) ? 32 : a.group;   // scaling granularity (K4: the 32-weight sub-block)
    const int GPC = KC / G;                         // groups (K4: sub-blocks) per unit
    uint8_t* xring = smem;
    uint8_t* cring = smem + PL::CODE_OFF;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PL::BAR_OFF);
    uint64_t* full = bars;                          // [XS] x tile landed
    uint64_t* empty = full + XS;                    // [XS] x tile consumed by the MMAs
    uint64_t* afull = empty + XS;                   // [NA] A buffer written by the dequant warps
    uint64_t* aempty = afull + NA;                  // [NA] A buffer consumed by the MMAs
    uint64_t* dfull = aempty + NA;                  // [DS] accumulator slot complete
    uint64_t* dempty = dfull + DS;                  // [DS] accumulator slot read by the epilogue
    uint64_t* ebar = dempty + DS;                   // epilogue rendezvous (all epilogue threads)
    uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(ebar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_smem + 1);
    unsigned int* ticket_smem = reinterpret_cast<unsigned int*>(tmem_base_smem + 2);
    uint32_t* nlut = reinterpret_cast<uint32_t*>(smem + PL::BAR_OFF + 1024);   // NF4: (hi | lo << 16) per code
    uint32_t* epi_ring = reinterpret_cast<uint32_t*>(smem + PL::EPI_OFF);   // [ring][256 threads][SWORDS]
    uint32_t* dq_ring = reinterpret_cast<uint32_t*>(smem + PL::DQ_OFF);     // [CS][8 warps][16][2]

    // the warp index broadcast from lane 0, so that the compiler knows it (and everything derived from
    // it: roles, tensor-memory addresses) to be the same across the warp
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = trange_begin(cta, a.U, a.P), u1 = trange_begin(cta + 1, a.U, a.P);

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int s = 0; s < XS; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], SPLIT ? 2 : 1); }
        for (int i = 0; i < NA; ++i) { mbar_init(&afull[i], TC_DQ_WARPS); mbar_init(&aempty[i], SPLIT ? 2 : 1); }
        for (int d = 0; d < DS; ++d) { mbar_init(&dfull[d], 1); mbar_init(&dempty[d], EW); }
        mbar_init(ebar, 32 * EW);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if constexpr (FMT == UQ_NF4) {
        // the codebook value c[q] as hi = bf16(c[q]) and lo = bf16(c[q] - hi): hi + lo carries 16 significant
        // bits of c[q] (relative error below 2^-16), so the MMAs multiply x by c[q] within that
        if (threadIdx.x < 16) {
            const float cq = reinterpret_cast<const float*>(a.zc)[threadIdx.x];
            const __nv_bfloat16 hi = __float2bfloat16_rn(cq);
            const __nv_bfloat16 lo = __float2bfloat16_rn(cq - __bfloat162float(hi));
            nlut[threadIdx.x] = (uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(lo) << 16);
        }
    }
    if (warp == 0) tmem_alloc(tmem_base_smem, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_smem;
    const uint32_t A_COL0 = 0;                      // A buffers: columns [0, 2*ACOLS)
    const uint32_t D_COL0 = NA * ACOLS;             // D slots: columns [NA*ACOLS, NA*ACOLS + DS*MPAD)

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer of x
        if (lane == 0) {
            auto issue_x = [&](int c, int s) {
                uint8_t* st = xring + s * XB;
#pragma unroll
                for (int q = 0; q < KC / 64; ++q)
                    tma_load_2d(st + q * (MPAD * 128), &tmap_x, c * KC + q * 64, 0, &full[s]);
            };
            // x may be written by the kernel before on the stream: loaded after the wait for it (the
            // dequant warps request the codes themselves)
            const int pre = (u1 - u0) < XS ? (int)(u1 - u0) : XS;
            const int CH = a.CH;
            int c = (int)(u0 % CH);
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int j = 0; j < pre; ++j) {
                mbar_arrive_expect_tx(&full[j], (uint32_t)XB);
                issue_x(c, j);
                if (++c == CH) c = 0;
            }
            int issued = pre;
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
                if (++c == CH) c = 0;
                if (++s == XS) s = 0;
            }
            // let the last copies land before the CTA can leave
            for (int j = issued - 1; j >= 0 && j >= issued - XS; --j)
                mbar_wait_bounded(&full[j % XS], (uint32_t)((j / XS) & 1), a.fault, FAULT_TC_WAIT);
        }
    } else if (warp == 1 || (NISS == 2 && warp == 2)) {
        // ---------------------------------------------------------------- MMA issuers
        // The whole warp runs the issue loop, so every operand (descriptors, tensor-memory columns,
        // ring positions) is computed once per warp as a warp-uniform value; one elected lane issues
        // the tcgen05.mma and tcgen05.commit instructions (a commit tracks the MMAs of the thread
        // that issues it, so the same lane issues both).  For Mpad <= 32 two warps issue: warp 1 the
        // CTA's even units (A buffer 0, accumulator slots [0, DH)), warp 2 the odd ones (A buffer 1,
        // slots [DH, 2 DH)).
        const int me = warp - 1, DH = DS / NISS;
        const bool leader = lane == 0;                   // the lane elect.sync picks in a converged warp
        int d = 0;
        uint32_t dph = 0;                                // phase of dempty[me * DH + d] (^1)
        const int KS = G / 16;                           // MMAs per group
        for (long long u = u0 + (SPLIT ? 0 : me); u < u1; u += (SPLIT ? 1 : NISS)) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const int i = (int)(u - u0);
            const int s = i % XS, ab = i % NA;
            const uint32_t sph = (uint32_t)((i / XS) & 1), aph = (uint32_t)((i / NA) & 1);
            bool ok = mbar_wait_bounded(&full[s], sph, a.fault, FAULT_TC_WAIT) &&
                      mbar_wait_bounded(&afull[ab], aph, a.fault, FAULT_TC_WAIT);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) { if (leader) *abort_flag = 1; break; }
            tc_fence_after();
            // B descriptors advance by 32 bytes per 16-k slice and by one x box (MPAD x 128 B)
            // per 64 k: the start-address field is byte address / 16
            const uint64_t bdesc0 = sw128_desc(xring + s * XB);
            const uint32_t acol0 = tmem + A_COL0 + ab * ACOLS;
            int ks = 0;
            for (int j = 0; j < GPC; ++j) {
                if (SPLIT && (j & 1) != me) { ks += KS; continue; }
                const int slot = me * DH + d;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&dempty[slot], dph ^ 1u, a.fault, FAULT_TC_WAIT));
                if (!ok) break;
                tc_fence_after();
                const uint32_t dcol = tmem + D_COL0 + slot * MPAD;
                for (int t = 0; t < KS; ++t) {
                    const int kk = ks + t;
                    const uint64_t bdesc = bdesc0 + (uint64_t)((kk >> 2) * (MPAD * 8) + (kk & 3) * 2);
                    mma_ts_elect(dcol, acol0 + kk * 8, bdesc, IDESC, t > 0 ? 1u : 0u);
                    if constexpr (TcFmt<FMT>::PLANES == 2)                 // NF4: the lo plane into the same sum
                        mma_ts_elect(dcol, acol0 + KC / 2 + kk * 8, bdesc, IDESC, 1u);
                }
                tc_commit_elect(&dfull[slot]);
                ks += KS;
                if (++d == DH) { d = 0; dph ^= 1u; }
            }
            if (!ok) { if (leader) *abort_flag = 1; break; }
            tc_commit_elect(&aempty[ab]);
            tc_commit_elect(&empty[s]);
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
        // Unit u's copies, CD units ahead, one cp.async group per unit: this warp's codes (16-row block
        // rb * 8 + rbl, the unit's CPU 512-byte chunks, contiguous in the fragment-order plane) into code
        // stage (u - u0) % CS, and the zero points of rows g and g + 8 (lanes c = 0, 1): INT4_ASYM's
        // nibble bytes, INT2_ASYM's fp16 zeros.
        constexpr int WB = TcFmt<FMT>::WBYTES, CPU = TcFmt<FMT>::CPU;
        constexpr int ZW = PL::ZW;
        auto issue_codes = [&](long long u) {
            if (u < u1) {
                const int rbc = (int)(u / a.CH), cc = (int)(u % a.CH);
                const int cs = (int)((u - u0) % CS);
                if (rbc * 8 + rbl < a.NB) {
                    const int ch0 = cc * CPU;                    // first chunk of the unit in the row block
                    const uint8_t* src = a.wq + (long long)(rbc * 8 + rbl) * 16 * a.rowbytes +
                                         (long long)(ch0 >> 4) * TILE_BYTES + (ch0 & 15) * CHUNK;
                    uint8_t* dst = cring + cs * TcFmt<FMT>::CODES + rbl * WB;
#pragma unroll
                    for (int q = 0; q < CPU; ++q) tc_cp_async16(dst + q * CHUNK + lane * 16, src + q * CHUNK + lane * 16);
                }
                if constexpr (ZW > 0) {
                    if (c4 < 2) {
                        const int r = g + 8 * c4;
                        const long long n = (long long)rbc * TC_ROWS + rbl * 16 + r;
                        const int Gn = a.K / G;
                        uint32_t* zdst = dq_ring + (cs * TC_DQ_WARPS + (warp - 4)) * 16 * ZW + r * ZW;
                        if (n < a.N) {
                            if constexpr (FMT == UQ_INT4_ASYM) {
                                const int ZB = (Gn + 1) >> 1;
                                stage_span(zdst, a.zc, n * ZB + (long long)cc * (GPC >> 1), GPC >> 1, (long long)a.N * ZB);
                            } else {
                                stage_span(zdst, a.zc, (n * Gn + (long long)cc * GPC) * 2, GPC * 2, (long long)a.N * Gn * 2);
                            }
                        }
                    }
                }
            }
            cp_async_commit();
        };
        // the first unit alone at first: requested together with the next CD - 1 units, its bytes would
        // arrive only with theirs; the others follow once it has landed
        issue_codes(u0);
        int ab = 0;
        uint32_t aph = 1;                               // aempty[] of the first round counts as free
        int rb = (int)(u0 / a.CH), c = (int)(u0 % a.CH);
        for (long long u = u0; u < u1; ++u) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            __syncwarp();                               // every lane is done with the stage refilled next
            const int cs = (int)((u - u0) % CS);
            // subtrahend per group as a bf16 pair: 128 + z (INT4_ASYM, INT2_ASYM), 128 + 8 (INT4_SYM), 128 (K4)
            constexpr int ZG = (FMT == UQ_INT4_ASYM || FMT == UQ_INT2_ASYM) ? KC / (16 * GB) : 1;   // groups per unit
            uint32_t zlo[ZG], zhi[ZG];
#pragma unroll
            for (int j = 0; j < ZG; ++j) zlo[j] = zhi[j] = (FMT == UQ_INT4_SYM) ? 0x43084308u : 0x43004300u;
            if (u == u0) {
                cp_async_wait<0>();                     // the first unit's codes (and zero words) landed
                __syncwarp();
                for (int j = 1; j <= CD; ++j) issue_codes(u0 + j);
            } else {
                issue_codes(u + CD);
                cp_async_wait<CD>();                    // unit u's codes (and zero words) landed
                __syncwarp();
            }
            if constexpr (ZW > 0) {
                const int Gn = a.K / G;
                const uint32_t* slot = dq_ring + (cs * TC_DQ_WARPS + (warp - 4)) * 16 * ZW;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const long long n = (long long)rb * TC_ROWS + rbl * 16 + g + 8 * h;
                    const uint32_t* zr = slot + (g + 8 * h) * ZW;
#pragma unroll
                    for (int j = 0; j < ZG; ++j) {
                        uint32_t z = 0;
                        if (n < a.N) {
                            if constexpr (FMT == UQ_INT4_ASYM) {
                                const int o = (int)((n * ((Gn + 1) >> 1) + (long long)c * (GPC >> 1)) & 3);
                                const uint64_t w = (uint64_t)zr[0] | ((uint64_t)zr[1] << 32);
                                z = (uint32_t)(w >> (8 * o + 4 * j)) & 15u;
                            } else {
                                // fp16 integer zero of group j: half (start parity) + j of the staged words
                                const int hi = (int)(((n * Gn + (long long)c * GPC) & 1) + j);
                                const uint16_t zh = (uint16_t)(zr[hi >> 1] >> (16 * (hi & 1)));
                                z = (uint32_t)half_bits_f32(zh);
                            }
                        }
                        const uint32_t zz = 0x43004300u | z | (z << 16);
                        if (h == 0) zlo[j] = zz; else zhi[j] = zz;
                    }
                }
            }
            bool ok = mbar_wait_bounded(&aempty[ab], aph, a.fault, FAULT_TC_WAIT);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) { *abort_flag = 1; break; }
            tc_fence_after();
            const uint8_t* rbase = cring + cs * TcFmt<FMT>::CODES + rbl * WB + lane * 16;
            const uint32_t acol = lane_addr + A_COL0 + ab * ACOLS;
            if constexpr (FMT == UQ_INT8_SYM) {
                // chunk q = 32 k = blocks 2q, 2q + 1; word 2b + h = row g + 8h, k 4c .. 4c + 3 of block b
#pragma unroll
                for (int q = 0; q < CPU; ++q) {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(rbase + q * CHUNK);
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
            } else if constexpr (FMT == UQ_INT2_ASYM) {
                // chunk q = 128 k = blocks 8q .. 8q + 7; word i holds blocks 2i (crumb pairs 0..3) and 2i + 1
                // (pairs 4..7), pair 4bb + pp laid out as the 4-bit pairs pp (0/2 row g, 1/3 row g + 8)
#pragma unroll
                for (int q = 0; q < CPU; ++q) {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(rbase + q * CHUNK);
                    const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int hs = 0; hs < 2; ++hs) {              // blocks 8q + 4hs .. + 3: one 16x256b x4 store
                        uint32_t v[16];
#pragma unroll
                        for (int b4 = 0; b4 < 4; ++b4) {
                            const int b = 4 * hs + b4;             // block within the chunk
                            const uint32_t wd = wv[b >> 1];
                            const int j = (8 * q + b) / GB;
                            uint32_t p0, p1, p2, p3;
                            if (b & 1) {
                                p0 = crumb_pair_lop3<4>(wd); p1 = crumb_pair_lop3<5>(wd);
                                p2 = crumb_pair_lop3<6>(wd); p3 = crumb_pair_lop3<7>(wd);
                            } else {
                                p0 = crumb_pair_lop3<0>(wd); p1 = crumb_pair_lop3<1>(wd);
                                p2 = crumb_pair_lop3<2>(wd); p3 = crumb_pair_lop3<3>(wd);
                            }
                            v[4 * b4 + 0] = bf16x2_sub(p0, zlo[j]);
                            v[4 * b4 + 1] = bf16x2_sub(p2, zlo[j]);
                            v[4 * b4 + 2] = bf16x2_sub(p1, zhi[j]);
                            v[4 * b4 + 3] = bf16x2_sub(p3, zhi[j]);
                        }
                        tmem_st_16x256b_x4(acol + (2 * q + hs) * 32, v);
                    }
                }
            } else if constexpr (FMT == UQ_NF4) {
                // chunk q = 64 k = blocks 4q .. 4q + 3, one word each; each code's codebook value as the bf16
                // pair (hi, lo) from the shared table: hi pairs into plane 0, lo pairs into plane 1
#pragma unroll
                for (int q = 0; q < CPU; ++q) {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(rbase + q * CHUNK);
                    const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
                    uint32_t vh[16], vl[16];
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
#pragma unroll
                        for (int P = 0; P < 4; ++P) {
                            const uint32_t e = nlut[(wv[b] >> (4 * P)) & 15u];
                            const uint32_t o = nlut[(wv[b] >> (16 + 4 * P)) & 15u];
                            const int slot = 4 * b + (P == 0 ? 0 : (P == 1 ? 2 : (P == 2 ? 1 : 3)));
                            vh[slot] = __byte_perm(e, o, 0x5410);
                            vl[slot] = __byte_perm(e, o, 0x7632);
                        }
                    }
                    tmem_st_16x256b_x4(acol + q * 32, vh);
                    tmem_st_16x256b_x4(acol + KC / 2 + q * 32, vl);
                }
            } else {
                // chunk q = 64 k = blocks 4q .. 4q + 3, one word each; pairs 0/2 are row g (k 4c, 4c+1 /
                // 4c+2, 4c+3), pairs 1/3 row g + 8
#pragma unroll
                for (int q = 0; q < CPU; ++q) {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(rbase + q * CHUNK);
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
            if (++ab == NA) { ab = 0; aph ^= 1u; }
            if (++c == a.CH) { c = 0; ++rb; }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // no copy lands after the CTA left
    } else if (warp >= 4 + TC_DQ_WARPS) {
        // ---------------------------------------------------------------- epilogue warps
        // Eight warps: warp 12 + e reads lane quarter e % 4 (rows 32 (e % 4) .. + 31, thread = row) and
        // columns [HW (e / 4), HW (e / 4) + HW) of every accumulator slot.
        asm volatile("griddepcontrol.wait;" ::: "memory");   // sx, workspace and y follow earlier work
        const int we = warp - 4 - TC_DQ_WARPS;
        const int quarter = we & 3, col0 = (we >> 2) * HW;
        const int r = quarter * 32 + lane;
        const int et = we * 32 + lane;                   // epilogue thread index
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t* er = epi_ring + et * SWORDS;           // this thread's slot (ring stride 256 * SWORDS)
        constexpr int RSTRIDE = 32 * EW * SWORDS;
        // this row's scale words (K4: its super-block record) staged TC_EPI_RING - 1 units ahead
        auto issue_scales = [&](long long u) {
            if (u < u1) {
                const int rbu = (int)(u / a.CH), cu = (int)(u % a.CH);
                const long long n = (long long)rbu * TC_ROWS + r;
                uint32_t* dst = er + (int)((u - u0) % TC_EPI_RING) * RSTRIDE;
                if (n < a.N) {
                    if constexpr (FMT == UQ_K4) {
                        tc_cp_async16(dst, a.scales + (n * (a.K >> 8) + cu) * 16);
                    } else {
                        const long long Gn = a.K / G;
                        stage_span(dst, a.scales, (n * Gn + (long long)cu * GPC) * 2, GPC * 2, (long long)a.N * Gn * 2);
                    }
                }
            }
            cp_async_commit();
        };
        for (int j = 0; j < TC_EPI_RING - 1; ++j) issue_scales(u0 + j);
        float acc[HW];
#pragma unroll
        for (int m = 0; m < HW; ++m) acc[m] = 0.f;
        // accumulator slots: unit u's groups are in the ring of the issuer that took it ((u - u0) mod
        // the issuer count), slots [DH * ring, DH * ring + DH), consumed in that issuer's order
        const int DH = DS / NISS;
        int dr0 = 0, dr1 = 0;                            // next slot of issuer ring 0 / 1
        uint32_t dp0 = 0u, dp1 = 0u, ephase = 0;         // and its phase
        // all epilogue threads meet here (bounded: returns false after the time limit)
        auto epi_sync = [&]() -> bool {
            mbar_arrive(ebar);
            const bool r_ok = mbar_wait_bounded(ebar, ephase, a.fault, FAULT_TC_WAIT);
            ephase ^= 1u;
            return r_ok;
        };
        const int first_rb = (int)(u0 / a.CH);
        int pend0 = -1, pend1 = -1;                      // row blocks whose partial sums this CTA stored
        int rb = first_rb, c = (int)(u0 % a.CH);
        for (long long u = u0; u < u1; ++u) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const int n = rb * TC_ROWS + r;
            const bool live = n < a.N;
            issue_scales(u + TC_EPI_RING - 1);
            cp_async_wait<TC_EPI_RING - 1>();
            const uint32_t* sw = er + (int)((u - u0) % TC_EPI_RING) * RSTRIDE;
            const int so = live ? (int)(((long long)n * (a.K / G) + (long long)c * GPC) & 1) : 0;   // halves
            bool ok = true;
            for (int j = 0; j < GPC; ++j) {
                // the issuer ring holding group j of unit u: SPLIT: j mod 2; alternate units: (u - u0) mod 2
                const int ring = SPLIT ? (j & 1) : (NISS == 2 ? (int)((u - u0) & 1) : 0);
                int d = ring ? dr1 : dr0;
                uint32_t dph = ring ? dp1 : dp0;
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
                float v[HW];
#pragma unroll
                for (int q = 0; q < HW / 8; ++q) tmem_ld8(lane_addr + D_COL0 + slot * MPAD + col0 + q * 8, &v[q * 8]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&dempty[slot]);
#pragma unroll
                for (int m = 0; m < HW; ++m) acc[m] = fmaf(s1, v[m], acc[m]);
                if (++d == DH) { d = 0; dph ^= 1u; }
                if (ring) { dr1 = d; dp1 = dph; } else { dr0 = d; dp0 = dph; }
                if constexpr (FMT == UQ_K4) {
                    const float* sx = a.sx + (long long)((c * KC + j * 32) >> 5) * MPAD + col0;
#pragma unroll
                    for (int m = 0; m < HW; ++m) acc[m] = fmaf(-s2, __ldg(sx + m), acc[m]);
                }
            }
            if (!ok) { *abort_flag = 1; break; }
            if (c == a.CH - 1 || u == u1 - 1) {
                // row block finished for this CTA: store y, or a partial and a ticket
                const bool fullcov = (c == a.CH - 1) && (rb != first_rb || (u0 % a.CH) == 0);
                if (fullcov) {
                    if (live)
#pragma unroll
                        for (int m = 0; m < HW; ++m)
                            if (col0 + m < a.M)
                                store_out(a, col0 + m, n, acc[m]);
                } else {
                    // partial sums of a row block shared with other CTAs: stored now, combined after the
                    // CTA's last unit (so the pipeline never waits on other CTAs mid-run)
                    const int pslot = 2 * cta + (rb == first_rb ? 0 : 1);
                    float* part = a.partials + (long long)pslot * TC_ROWS * MPAD + r;   // [slot][m][row]
#pragma unroll
                    for (int m = 0; m < HW; ++m) part[(col0 + m) * TC_ROWS] = acc[m];
                    if (pend0 < 0) pend0 = rb; else pend1 = rb;
                }
#pragma unroll
                for (int m = 0; m < HW; ++m) acc[m] = 0.f;
            }
            if (++c == a.CH) { c = 0; ++rb; }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        // Row blocks shared with other CTAs: every contributor makes its partial sums visible, then takes
        // a ticket; the last one sums all contributors' partials in CTA order (fixed, so the result is
        // deterministic) and writes y.  Nobody waits for another CTA.
        if (pend0 >= 0 && !__shfl_sync(0xffffffffu, *abort_flag, 0)) {
            __threadfence();
            bool ok = epi_sync();
            if (ok && et == 0) {
                ticket_smem[0] = atomicAdd(a.tickets + pend0, 1u);
                if (pend1 >= 0) ticket_smem[1] = atomicAdd(a.tickets + pend1, 1u);
            }
            ok = ok && epi_sync();
            for (int k = 0; ok && k < 2; ++k) {
                const int prb = k ? pend1 : pend0;
                if (prb < 0) continue;
                const unsigned int old = ticket_smem[k];
                const long long uf = (long long)prb * a.CH;
                const int cf = tworker_of(uf, a.U, a.P), cl = tworker_of(uf + a.CH - 1, a.U, a.P);
                if (old != (unsigned int)(cl - cf)) continue;
                __threadfence();
#pragma unroll
                for (int m = 0; m < HW; ++m) acc[m] = 0.f;
                for (int c2 = cf; c2 <= cl; ++c2) {
                    const int rb2 = (int)(trange_begin(c2, a.U, a.P) / a.CH);
                    const int slot2 = 2 * c2 + (prb == rb2 ? 0 : 1);
                    const float* p2 = a.partials + (long long)slot2 * TC_ROWS * MPAD + r;
#pragma unroll
                    for (int m = 0; m < HW; ++m) acc[m] += __ldcg(p2 + (col0 + m) * TC_ROWS);
                }
                const int n = prb * TC_ROWS + r;
                if (n < a.N)
#pragma unroll
                    for (int m = 0; m < HW; ++m)
                        if (col0 + m < a.M)
                            store_out(a, col0 + m, n, acc[m]);
                if (et == 0) a.tickets[prb] = 0u;
            }
            if (!ok) *abort_flag = 1;
        }
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
        cfg.blockDim = dim3(tc_threads(MPAD));
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
        tc_kernel<FMT, MPAD, GB><<<grid, tc_threads(MPAD), smem, st>>>(mx, a);
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
    if constexpr (FMT != UQ_K4) {
        switch (a.group) {
            case 32: return launch_tc_mg<FMT, 2>(mpad, mx, a, smem, grid, st);
            case 64: return launch_tc_mg<FMT, 4>(mpad, mx, a, smem, grid, st);
            case 128: return launch_tc_mg<FMT, 8>(mpad, mx, a, smem, grid, st);
            default: return cudaErrorInvalidValue;
        }
    } else {
        return launch_tc_mg<FMT, 2>(mpad, mx, a, smem, grid, st);
    }
}
}  // namespace

bool tc_supported(int fmt, int N, int K) {
    if (fmt < UQ_INT4_SYM || fmt > UQ_K4) return false;
    if (N < 1 || K % fmt_kt(fmt)) return false;
    return encode_fn() != nullptr;
}

namespace {
template <int FMT, int GB>
size_t tc_smem_fg(int mpad) {
    switch (mpad) {
        case 16: return TcPlan<FMT, 16, GB>::SMEM;
        case 32: return TcPlan<FMT, 32, GB>::SMEM;
        case 48: return TcPlan<FMT, 48, GB>::SMEM;
        case 64: return TcPlan<FMT, 64, GB>::SMEM;
        default: return 0;
    }
}
template <int FMT>
size_t tc_smem_fmt(int mpad, int group) {
    if (FMT == UQ_K4) return tc_smem_fg<FMT, 2>(mpad);
    switch (group) {
        case 32: return tc_smem_fg<FMT, 2>(mpad);
        case 64: return tc_smem_fg<FMT, 4>(mpad);
        case 128: return tc_smem_fg<FMT, 8>(mpad);
        default: return 0;
    }
}
}  // namespace

int tc_plan(int fmt, int mpad, int group, size_t* smem) {
    size_t b = 0;
    switch (fmt) {
        case UQ_INT4_SYM: b = tc_smem_fmt<UQ_INT4_SYM>(mpad, group); break;
        case UQ_INT4_ASYM: b = tc_smem_fmt<UQ_INT4_ASYM>(mpad, group); break;
        case UQ_INT8_SYM: b = tc_smem_fmt<UQ_INT8_SYM>(mpad, group); break;
        case UQ_INT2_ASYM: b = tc_smem_fmt<UQ_INT2_ASYM>(mpad, group); break;
        case UQ_NF4: b = tc_smem_fmt<UQ_NF4>(mpad, group); break;
        case UQ_K4: b = tc_smem_fmt<UQ_K4>(mpad, group); break;
        default: return -1;
    }
    if (!b) return -1;
    *smem = b;
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
        case UQ_INT2_ASYM: return launch_tc_m<UQ_INT2_ASYM>(a.Mpad, mx, a, smem, grid, st);
        case UQ_NF4: return launch_tc_m<UQ_NF4>(a.Mpad, mx, a, smem, grid, st);
        case UQ_K4: return launch_tc_m<UQ_K4>(a.Mpad, mx, a, smem, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace uq
