// uq_common.cuh -- packed layout, format traits and PTX helpers shared by the uq kernels (sm_103a).
//
// Packed code plane ("pack multiple low-bit values into bytes", "Ultra LLM Engine",
// section "Quantization"): the N x K code matrix is cut into tiles of RB = 8 rows by
// 512 bytes of codes (KT = 4096 / bits codes).  The last tile of each row block is
// narrower when K is not a multiple of KT, the last row block shorter when N is not
// a multiple of 8.  Each tile is stored contiguously (row-major inside), the tiles
// of a row block one after another in k order, the row blocks one after another:
//
//     tile(nb, kb) = nb * 8 * rowbytes + rows(nb) * kb * 512,   rowbytes = K * bits / 8
//
// so one bulk copy fetches one tile.  Inside a tile row, 32-bit words are in natural
// k order; inside a word the codes are permuted so that a shift and a mask put two
// k-consecutive codes into the two halves of a register:
//     4-bit: code 2p at bits [4p, 4p+4), code 2p+1 at bits [16+4p, 16+4p+4)   (p = 0..3)
//     2-bit: code 2p at bits [2p, 2p+2), code 2p+1 at bits [16+2p, 16+2p+2)   (p = 0..7)
//     8-bit: code i at bits [8i, 8i+8)
// Signed formats are stored biased: INT4_SYM as q + 8, INT8_SYM as q + 128.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/uq.h"

namespace uq {

constexpr int RB = 8;            // rows per tile
constexpr int SLICE = 512;       // bytes of codes per row of a full tile
constexpr int TILE_BYTES = RB * SLICE;

__host__ __device__ constexpr int fmt_bits(int fmt) {
    return fmt == UQ_INT8_SYM ? 8 : (fmt == UQ_INT2_ASYM ? 2 : 4);
}
__host__ __device__ constexpr int fmt_kt(int fmt) { return 4096 / fmt_bits(fmt); }     // codes per tile row
__host__ __device__ constexpr int fmt_cpl(int fmt) { return 128 / fmt_bits(fmt); }     // codes per 16-byte lane chunk
__host__ __device__ constexpr int fmt_cpw(int fmt) { return 32 / fmt_bits(fmt); }      // codes per 32-bit word
__host__ __device__ constexpr int fmt_bias(int fmt) {
    return fmt == UQ_INT4_SYM ? 8 : (fmt == UQ_INT8_SYM ? 128 : 0);
}

// Bit position of code i (0 <= i < codes per word) inside its 32-bit word.
__host__ __device__ inline int code_bitpos(int bits, int i) {
    if (bits == 8) return 8 * i;
    return (i & 1) ? 16 + bits * (i >> 1) : bits * (i >> 1);
}

// Geometry of one weight matrix in the packed layout.
struct Layout {
    int N, K, bits, KT;
    int NB, KB;              // row blocks, k tiles
    long long rowbytes;      // K * bits / 8

    __host__ __device__ Layout(int n, int k, int fmt)
        : N(n), K(k), bits(fmt_bits(fmt)), KT(fmt_kt(fmt)),
          NB((n + RB - 1) / RB), KB((k + fmt_kt(fmt) - 1) / fmt_kt(fmt)),
          rowbytes((long long)k * fmt_bits(fmt) / 8) {}

    __host__ __device__ int rows(int nb) const { int r = N - nb * RB; return r < RB ? r : RB; }
    __host__ __device__ int width(int kb) const { int w = K - kb * KT; return w < KT ? w : KT; }
    __host__ __device__ int slice_bytes(int kb) const { return width(kb) * bits / 8; }
    __host__ __device__ long long tile_offset(int nb, int kb) const {
        return (long long)nb * RB * rowbytes + (long long)rows(nb) * kb * SLICE;
    }
    // byte offset of the 32-bit word holding code k of row n
    __host__ __device__ long long word_offset(int n, int k) const {
        int nb = n / RB, r = n % RB, kb = k / KT, kk = k % KT;
        return tile_offset(nb, kb) + (long long)r * slice_bytes(kb) + (long long)(kk / (32 / bits)) * 4;
    }
};

// ---------------------------------------------------------------------------------------------
// Unpacking (shared by the debug exports and the GEMV/GEMM kernels).
// A bf16 with biased exponent 134 (0x43) and a 7-bit mantissa m equals 128 + m exactly, so
// OR-ing a small code into the mantissa field of 0x4300 yields 128 + code without a conversion.

// bf16x2 (128 + code[2p], 128 + code[2p+1]) from a 4-bit word
__device__ __forceinline__ uint32_t nib_pair_bf16(uint32_t w, int p) {
    return ((w >> (4 * p)) & 0x000F000Fu) | 0x43004300u;
}
// bf16x2 (128 + code[2p], 128 + code[2p+1]) from a 2-bit word
__device__ __forceinline__ uint32_t crumb_pair_bf16(uint32_t w, int p) {
    return ((w >> (2 * p)) & 0x00030003u) | 0x43004300u;
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
// Bounded wait: polls until the phase with `parity` completes or WAIT_LIMIT_NS of wall time
// (the %globaltimer nanosecond clock) have passed; then records `code` in the fault word and
// returns false so the caller can leave instead of hanging the GPU.
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
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > WAIT_LIMIT_NS) break;
    }
    atomicOr(fault, code);
    return false;
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

}  // namespace uq
