// uq_common.cuh -- packed layout, format traits and PTX helpers shared by the uq kernels (sm_103a).
//
// Packed code plane ("pack multiple low-bit values into bytes", "Ultra LLM Engine", section
// "Quantization"), laid out for the warp-level tensor-core instruction mma.m16n8k16:
//
//  * Rows are taken in blocks of 16 (N is padded to Np = a multiple of 16), k in chunks of
//    kc codes (kc = 64 for 4-bit, 128 for 2-bit, 32 for 8-bit; K is padded to Kp, a multiple
//    of kc).  A chunk of one row block is 512 bytes: 32 lanes x 16 bytes.
//  * A tile is 16 rows x KT codes (KT = 1024 / 2048 / 512 codes = 16 chunks = 8 KB); the last
//    tile of a row block is narrower when Kp is not a multiple of KT.  Tiles of a row block
//    follow each other in k order, row blocks follow each other:
//        tile(nb, kb) = nb * 16 * Kp * bits/8 + kb * 8192.
//  * Inside a chunk, lane L = 4g + c (g = 0..7, c = 0..3) holds, for every 16-wide k block,
//    the codes of rows g and g + 8 at k = 16b + 4c .. 16b + 4c + 3 -- exactly the A-operand
//    fragment that thread L feeds to mma.m16n8k16 (with the k slots of the instruction mapped
//    to 4c..4c+3, a permutation the B operand repeats).  For 4-bit codes one 32-bit word is
//    one k block: pair p (p = 0..3) sits at bits [4p, 4p+4) (even k) and [16+4p, 20+4p) (odd k),
//    with p = h + 2*(j >> 1) for row g + 8h and k = 16b + 4c + j: a shift and a mask give the
//    bf16 pair of register a_p.  2-bit words hold two k blocks (pairs 0..3 and 4..7 at 2-bit
//    fields); 8-bit words hold the 4 codes of one row (word 2*b' + h of the chunk, b' = block).
//  * Signed formats are stored biased: INT4_SYM as q + 8, INT8_SYM as q + 128.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/uq.h"

namespace uq {

constexpr int RB = 16;           // rows per row block (the M of mma.m16n8k16)
constexpr int CHUNK = 512;       // bytes of one k chunk of a row block
constexpr int TILE_BYTES = 8192; // a full tile: 16 chunks

__host__ __device__ constexpr int fmt_bits(int fmt) {
    return fmt == UQ_INT8_SYM ? 8 : (fmt == UQ_INT2_ASYM ? 2 : 4);
}
__host__ __device__ constexpr int fmt_kt(int fmt) { return 4096 / fmt_bits(fmt); }        // codes per tile row
__host__ __device__ constexpr int fmt_kc(int fmt) { return CHUNK * 8 / fmt_bits(fmt) / RB; }   // codes per chunk row
__host__ __device__ constexpr int fmt_cpw(int fmt) { return 32 / fmt_bits(fmt); }            // codes per 32-bit word
__host__ __device__ constexpr int fmt_bias(int fmt) {
    return fmt == UQ_INT4_SYM ? 8 : (fmt == UQ_INT8_SYM ? 128 : 0);
}

// Geometry of one weight matrix in the packed layout.
struct Layout {
    int N, K, bits, KT, kc, Np, Kp, NB, KB;
    long long rowbytes;      // Kp * bits / 8

    __host__ __device__ Layout(int n, int k, int fmt)
        : N(n), K(k), bits(fmt_bits(fmt)), KT(fmt_kt(fmt)), kc(fmt_kc(fmt)),
          Np((n + RB - 1) / RB * RB), Kp((k + fmt_kc(fmt) - 1) / fmt_kc(fmt) * fmt_kc(fmt)),
          NB((n + RB - 1) / RB), KB(0), rowbytes(0) {
        KB = (Kp + KT - 1) / KT;
        rowbytes = (long long)Kp * bits / 8;
    }
    __host__ __device__ long long bytes() const { return (long long)Np * rowbytes; }
    __host__ __device__ int width(int kb) const { int w = Kp - kb * KT; return w < KT ? w : KT; }
    __host__ __device__ int chunks(int kb) const { return width(kb) / kc; }
    __host__ __device__ int tile_bytes(int kb) const { return chunks(kb) * CHUNK; }
    __host__ __device__ long long tile_offset(int nb, int kb) const {
        return (long long)nb * RB * rowbytes + (long long)kb * TILE_BYTES;
    }
    // Row and k of code slot `s` of the 32-bit word at byte offset `off` (a multiple of 4).
    // Slots: 4-bit s = 2p + hi (p = pair 0..3), 2-bit s = 2p + hi (p = 0..7), 8-bit s = byte.
    __host__ __device__ void slot_nk(long long off, int s, int* n, int* k) const {
        const long long rbb = (long long)RB * rowbytes;
        const int nb = (int)(off / rbb);
        const long long rem = off % rbb;
        const int kb = (int)(rem / TILE_BYTES);
        const int rem2 = (int)(rem % TILE_BYTES);
        const int q = rem2 / CHUNK, L = (rem2 % CHUNK) / 16, i = (rem2 % 16) / 4;
        const int g = L >> 2, c = L & 3;
        const int k0 = kb * KT + q * kc;
        int r = 0, kk = 0;
        if (bits == 4) {
            const int p = s >> 1, hi = s & 1;
            r = 8 * (p & 1) + g;
            kk = i * 16 + 4 * c + 2 * (p >> 1) + hi;
        } else if (bits == 2) {
            const int p = s >> 1, hi = s & 1, bb = p >> 2, pp = p & 3;
            r = 8 * (pp & 1) + g;
            kk = (2 * i + bb) * 16 + 4 * c + 2 * (pp >> 1) + hi;
        } else {
            r = 8 * (i & 1) + g;
            kk = (i >> 1) * 16 + 4 * c + s;
        }
        *n = nb * RB + r;
        *k = k0 + kk;
    }
};

// bit position of code slot s inside its word (see Layout::slot_nk)
__host__ __device__ inline int slot_bitpos(int bits, int s) {
    if (bits == 8) return 8 * s;
    const int p = s >> 1, hi = s & 1;
    return bits * p + 16 * hi;
}

// ---------------------------------------------------------------------------------------------
// Unpacking (shared by the debug exports and the GEMV/GEMM kernels).
// A bf16 with biased exponent 134 (0x43) and a 7-bit mantissa m equals 128 + m exactly, so
// OR-ing a small code into the mantissa field of 0x4300 yields 128 + code without a conversion.

// bf16x2 (128 + code) of nibble pair P (bits 4P.. of each half) / crumb pair P (bits 2P..): one
// lop3 ((w & mask) | magic), after a shift unless P == 0
template <int P>
__device__ __forceinline__ uint32_t nib_pair_lop3(uint32_t w) {
    uint32_t r;
    if constexpr (P == 0) {
        asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(r) : "r"(w));
    } else {
        asm("{\n\t.reg .b32 t;\n\tshr.b32 t, %1, %2;\n\tlop3.b32 %0, t, 0x000F000F, 0x43004300, 0xEA;\n\t}"
            : "=r"(r) : "r"(w), "n"(4 * P));
    }
    return r;
}
template <int P>
__device__ __forceinline__ uint32_t crumb_pair_lop3(uint32_t w) {
    uint32_t r;
    if constexpr (P == 0) {
        asm("lop3.b32 %0, %1, 0x00030003, 0x43004300, 0xEA;" : "=r"(r) : "r"(w));
    } else {
        asm("{\n\t.reg .b32 t;\n\tshr.b32 t, %1, %2;\n\tlop3.b32 %0, t, 0x00030003, 0x43004300, 0xEA;\n\t}"
            : "=r"(r) : "r"(w), "n"(2 * P));
    }
    return r;
}
// fp32 (2^23 + byte i of w): a float with biased exponent 150 and the byte in the mantissa
__device__ __forceinline__ float byte_magic_f32(uint32_t w, int i) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, (unsigned)(i | 0x7540)));
}
__device__ __forceinline__ float bf16lo_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// fp32 from an fp16 bit pattern (exact, subnormals included)
__device__ __forceinline__ float half_bits_f32(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

// Two chained mixed-precision FMAs, low halves first: d = (c + a.lo*b.lo) + a.hi*b.hi, each
// fma.rn.f32.bf16 rounding once to fp32 (bf16 x bf16 products are exact in fp32).
__device__ __forceinline__ float fma2_bf16(uint32_t a2, uint32_t b2, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %3;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    return d;
}

// ---------------------------------------------------------------------------------------------
// PTX wrappers: mbarrier, bulk async copy, proxy fences.

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// raise the transaction count of the current phase without arriving (the phase cannot complete
// before its expected arrivals, so a copy issued now may be counted before its arrival comes)
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// The same test, but a thread whose phase is not complete is suspended in the instruction until
// the phase completes or up to `ns` nanoseconds pass, instead of returning at once: a waiting warp
// then leaves its issue slots to the working ones rather than spinning.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(ns) : "memory");
    return ok != 0;
}
// Bounded wait: waits until the phase with `parity` completes or WAIT_LIMIT_NS of wall time
// (the %globaltimer nanosecond clock) have passed; then records `code` in the fault word and
// returns false so the caller can leave instead of hanging the GPU.  Each attempt may suspend the
// thread for up to 1 us (woken early when the phase completes).
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;   // 2 s
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned int* fault,
                                                  unsigned int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_sleep(bar, parity, 1000u))
        if (global_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(fault, code);
            return false;
        }
    return true;
}
// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// fault codes written to the device fault word
constexpr unsigned int FAULT_GEMV_WAIT = 1u;
constexpr unsigned int FAULT_TC_WAIT = 2u;
constexpr unsigned int FAULT_GEMV_SPLIT = 4u;   // a launch's work split exceeded what the kernel holds
constexpr unsigned int FAULT_ROPE_POS = 8u;     // a row's position lay outside the rope table (row not written)

}  // namespace uq
