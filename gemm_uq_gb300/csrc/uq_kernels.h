// uq_kernels.h -- internal declarations shared by the uq CUDA sources and the C-ABI host code.
#pragma once

#include "uq_common.cuh"

namespace uq {

// records the message uq_last_error() returns on the calling thread (uq_api.cu)
void set_last_error(const char* msg);
// whether GEMV kernels are launched with programmatic dependent launch (uq_set_launch_overlap)
bool launch_overlap();

// reads and clears the fault word of uq_gemm_noalloc launches on the current device (uq_noalloc.cu)
cudaError_t noalloc_take_fault(unsigned int* v);

// offline kernels (uq_pack.cu)
cudaError_t launch_pack(int fmt, const int8_t* codes, uint8_t* wq, int N, int K, unsigned int* bad,
                        cudaStream_t st);
cudaError_t launch_unpack(int fmt, const uint8_t* wq, int8_t* codes, int N, int K, cudaStream_t st);
cudaError_t launch_pack_gguf(int qtype, const uint8_t* blocks, uint8_t* wq, uint16_t* scales, int N, int K,
                             cudaStream_t st);   // qtype 0 = Q4_0, 1 = Q8_0
cudaError_t launch_dequant(int fmt, const uint8_t* wq, const uint8_t* scales, const uint8_t* zc, float* w,
                           int N, int K, int group, cudaStream_t st);
cudaError_t launch_pack_kmeta(const uint16_t* d, const uint16_t* dmin, const uint8_t* sc, const uint8_t* m,
                              uint8_t* meta, long long count, unsigned int* bad, cudaStream_t st);
cudaError_t launch_pack_zeros(const uint8_t* z, uint8_t* out, int N, int G, cudaStream_t st);
cudaError_t launch_quantize(int fmt, const float* w, int8_t* codes, uint16_t* scales, void* zeros,
                            const float* codebook, int N, int K, int group, cudaStream_t st);
cudaError_t launch_quantize_k4(const float* w, int8_t* codes, uint16_t* d, uint16_t* dmin, uint8_t* sc,
                               uint8_t* m, int N, int K, cudaStream_t st);

// fused RMSNorm + RoPE and its cos/sin table (uq_norm.cu)
cudaError_t launch_rope_table(float* table, int max_pos, int head_dim, double base, cudaStream_t st);
cudaError_t launch_rmsnorm_rope(const uint16_t* x, const uint16_t* gamma, const int32_t* pos, const float* table,
                                uint16_t* y, int M, int D, int head_dim, int max_pos, float eps, unsigned int* fault,
                                int sms, cudaStream_t st);

// small-M GEMV (uq_gemv.cu)
struct GemvArgs {
    const uint16_t* x;        // bf16 [M][ldx]
    const uint8_t* wq;        // packed codes
    const uint8_t* scales;    // fp16 [N][K/group] or K4 records
    const uint8_t* zc;        // zeros / codebook / NULL
    uint16_t* y;              // bf16 [M][ldy]
    int M, N, K, group, ldx, ldy;
    int NB, KB;               // row blocks, k tiles
    long long T;              // tiles = NB * KB
    int P;                    // workers that split the tiles, P <= T: warps (CUDA-core GEMV, W4A8) or
                              // CTAs (mma GEMV)
    float* partials;          // fp32 split-K partial sums: [T][16][M] (mma and W4A8 GEMVs, summed by the
                              // second pass), [2P][16][M] (CUDA-core GEMV: first and last row block of
                              // each worker)
    unsigned int* tickets;    // [NB], zero between calls
    unsigned int* fault;      // device fault word
    int overlap;              // launched with programmatic stream serialization (set by the launcher)
    int cta_rows;             // mma / W4A8 GEMV: > 0 = every CTA owns whole row blocks (combined in shared
                              // memory, no second pass; mma GEMV: the most tiles a CTA gets);
                              // 0 = workers split row blocks anywhere (second pass)
    float* out32;             // gate pass of the gated projection: fp32 results [M][ldy] instead of y
    const float* gate32;      // up pass: y = bf16(silu(gate32) * result), gate32 [M][ldy] fp32
    int gated;                // mma GEMV only: the gated projection in one launch; (wq, scales, zc) are the
                              // gate weight, (wq2, scales2, zc2) the up weight, NB and T count both
    const uint8_t* wq2;
    const uint8_t* scales2;
    const uint8_t* zc2;
    int a8;                   // the W4A8 GEMV (integer x codes):
    const int8_t* xq;         //   x codes [M][Kpq], each 32 k in the integer mma's B fragment order
    const float* sxq;         //   per-row scales of x [M]
    const int* sxl;           //   per (row, group) sums of the codes [M][ceil(Kpq / group)]
    int Kpq;                  //   bytes per row of xq
    int ring_slots;           // mma GEMV: ring slots and x-sum table groups of the launch (set by its launcher)
    int sx_groups;
    int mma_pairs;            // mma GEMV: pairs of compute warps that take tiles (set by its launcher)
};
// formats whose GEMV runs on mma.sync (all six)
inline bool gemv_is_mma(int fmt) {
    return fmt == UQ_INT4_SYM || fmt == UQ_INT4_ASYM || fmt == UQ_INT2_ASYM || fmt == UQ_K4 || fmt == UQ_INT8_SYM ||
           fmt == UQ_NF4;
}
// formats of the mma.sync GEMM (gemm_mma_kernel: 9..64 rows)
inline bool gemm_mma_format(int fmt) {
    return fmt == UQ_INT4_SYM || fmt == UQ_INT4_ASYM || fmt == UQ_INT2_ASYM || fmt == UQ_K4;
}
// Plans one GEMV launch from its shape fields (M, N, K, group, NB, KB, T, gated, a8) and the SM
// count: sets a.P and a.cta_rows.  Returns the grid, or 0 when no plan fits (K too long for the
// kernel's shared memory at this M).
int gemv_plan(GemvArgs& a, int fmt, int sms);
// what a planned launch needs: fp32 partial-sum floats, the per-row-block tickets, kernel launches
size_t gemv_partials_floats(int fmt, const GemvArgs& a);
bool gemv_uses_tickets(int fmt, const GemvArgs& a);
int gemv_launches(int fmt, const GemvArgs& a);
cudaError_t launch_gemv(int fmt, const GemvArgs& a, int grid, cudaStream_t st);
// the second pass of a stream-K split (tile partial sums [T][16][M] summed in k order)
cudaError_t launch_gemv_second_pass(const GemvArgs& a, int sms, cudaStream_t st);

// batched decode on mma.sync for the 4-bit and 2-bit formats, 9 <= M <= 64 (uq_gemm_mma.cu)
struct GemmArgs {
    const uint16_t* x;        // bf16 [M][ldx]
    const uint8_t* wq;        // packed codes
    const uint8_t* scales;    // fp16 [N][K/group] or K4 records
    const uint8_t* zc;        // INT4_ASYM zero nibbles, INT2_ASYM fp16 zeros, else NULL
    uint16_t* y;              // bf16 [M][ldy]
    int M, N, K, group, ldx, ldy;
    int NB;                   // row blocks of 16
    int UB;                   // k units per row (4 chunks of codes each)
    int KS;                   // k splits: CTAs per row group of 8 row blocks
    const float* sx;          // K4: column sums of x per 32-k block [K/32][Mpad], else NULL
    int Mpad;                 // columns of sx (8 x column blocks)
    float* partials;          // KS > 1: [KS][NB * 16][M] fp32
    float* out32;             // gate pass of the gated projection: fp32 results [M][ldy] instead of y
    const float* gate32;      // up pass: y = bf16(silu(gate32) * result)
};
int gemm_mma_units(int fmt, int K);               // k units per row
int gemm_mma_splits(int NB, int UB, int sms);     // k splits per row group
// the kernel, then (KS > 1) the second pass over the splits
cudaError_t launch_gemm_mma(int fmt, const GemmArgs& a, int sms, cudaStream_t st);

// W4A8 / W8A8 (uq_w4a8.cu): x codes and scales, then the integer GEMV
cudaError_t launch_quant_x(const uint16_t* x, int8_t* xq, float* sx, int* sxl, int M, int K, int Kp, int gs, int perm,
                           cudaStream_t st);
cudaError_t launch_gemv_a8(int fmt, const GemvArgs& a, const int8_t* xq, const float* sxs, const int* sxl, int Kp,
                           int grid, cudaStream_t st);


// tensor-core GEMM for M >= 16 (uq_tc.cu)
struct TcArgs {
    const uint8_t* wq;        // packed codes
    long long rowbytes;       // bytes of one padded row of codes
    int NB;                   // row blocks of 16
    const uint8_t* scales;    // fp16 [N][K/group] or K4 records
    const uint8_t* zc;        // INT4_ASYM zero nibbles, else NULL
    uint16_t* y;              // bf16 [M][ldy]
    const float* sx;          // K4: column sums of x per 32-k block [K/32][Mpad], else NULL
    int M, Mpad, N, K, group, ldx, ldy;
    int CH;                   // units (chunks of 128 code bytes) per 128-row block
    long long U;              // units = ceil(N/128) * CH
    int P;                    // CTAs, P <= U
    float* partials;          // [2P][128][Mpad]
    unsigned int* tickets;    // [ceil(N/128)]
    unsigned int* fault;
    float* out32;             // gate pass of the gated projection: fp32 results [M][ldy] instead of y
    const float* gate32;      // up pass: y = bf16(silu(gate32) * result)
};

// silu(g) * u in fp32 (silu(g) = g / (1 + e^-g)), the gated projection's epilogue
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// The one place every kernel writes an output element (row m of x, output column n): bf16 y; or, for
// the gated projection, fp32 g (the gate pass) or bf16 silu(g) * u (the up pass; the product in fp32,
// one rounding to bf16).
template <class Args>
__device__ __forceinline__ void store_out(const Args& a, int m, int n, float v) {
    const long long idx = (long long)m * a.ldy + n;
    if (a.out32) {
        a.out32[idx] = v;
        return;
    }
    if (a.gate32) v = silu_mul(a.gate32[idx], v);
    a.y[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
bool tc_supported(int fmt, int N, int K);
int tc_plan(int fmt, int mpad, int group, size_t* smem);   // dynamic shared memory of the launch
cudaError_t launch_colsum32(const uint16_t* x, float* sx, int M, int mpad, int K, int ldx, cudaStream_t st);
cudaError_t launch_tc(int fmt, const uint16_t* x, const TcArgs& a, size_t smem, int grid, cudaStream_t st);

}  // namespace uq
