/*
 * uq.h -- C ABI of the group-wise weight-only quantized decode GEMV/GEMM library (sm_103a).
 *
 * What the library computes ("Ultra LLM Engine", section "Fused Kernels": a
 * dequantized-weight GEMV for single-token decode and a dequantized-weight GEMM
 * for batched decode; section "Quantization": group-wise INT-N and NormalFloat4
 * weights that are packed into bytes and dequantized by the fused kernels):
 *
 *     y[m][n] = bf16_RNE( sum_k x[m][k] * W_hat[n][k] ),   fp32 accumulation,
 *
 * where x is M x K bf16, W_hat is the N x K dequantized weight (a linear layer's
 * weight, K contiguous) and y is M x N bf16.  W_hat is never materialised: the
 * kernels stream packed codes from HBM and unpack them in registers, where they feed
 * warp-level mma.sync instructions (4-bit and 2-bit formats: M <= 15, and K4 at any M; INT8 and
 * NF4: M <= 15), or are written as the integer part of the weights straight
 * into tensor memory as the A operand of tcgen05 tensor-core MMAs (M >= 16 otherwise); per-group
 * scales are applied to fp32 group sums.
 *
 * Weight formats (g = group size along K):
 *   UQ_INT4_SYM   codes q in [-8, 7],  fp16 scale s per group        W_hat = s*q
 *   UQ_INT4_ASYM  codes q in [0, 15],  fp16 s + 4-bit zero z         W_hat = s*(q - z)
 *   UQ_INT8_SYM   codes q in [-128,127] fp16 s per group             W_hat = s*q
 *   UQ_INT2_ASYM  codes q in [0, 3],   fp16 s + fp16 z (integer)     W_hat = s*(q - z)
 *   UQ_NF4        codes q in [0, 15],  fp16 absmax a, fp32 c[16]     W_hat = RN32(a*c[q])
 *   UQ_K4         codes q in [0, 15],  256-weight super-blocks of 8 x 32: fp16 d, dmin,
 *                 6-bit sc_j, m_j per 32-weight sub-block             W_hat = RN32(d*sc_j*q - dmin*m_j)
 *
 * Conventions for every call:
 *   - Pointers marked (device) are CUDA device memory owned by the caller; the
 *     library never frees or retains them.  Pointers must be 16-byte aligned
 *     (else UQ_ERR_ALIGN).  bf16 and fp16 arrays are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Calls are asynchronous and stream-ordered unless stated otherwise.
 *   - Errors are returned, never raised: no exception crosses the ABI, no kernel
 *     traps or asserts, and there is no silent fallback to another implementation.
 *   - The library runs on the device that is current on the calling thread.
 */
#ifndef UQ_H
#define UQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum uq_status {
    UQ_OK = 0,
    UQ_ERR_INVALID = 1,      /* bad argument: size, null pointer, code out of range, metadata mismatch */
    UQ_ERR_UNSUPPORTED = 2,  /* valid request outside what the kernels implement (group, K multiple, arch) */
    UQ_ERR_ALIGN = 3,        /* a pointer is not 16-byte aligned */
    UQ_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    UQ_ERR_NOMEM = 5         /* library-owned workspace could not be allocated (or not during capture) */
} uq_status;

typedef enum uq_fmt {
    UQ_INT4_SYM = 0,
    UQ_INT4_ASYM = 1,
    UQ_INT8_SYM = 2,
    UQ_INT2_ASYM = 3,
    UQ_NF4 = 4,
    UQ_K4 = 5
} uq_fmt;

/* GGUF block types uq_pack_gguf reads (the GGUF file format's block layouts). */
typedef enum uq_gguf_type {
    UQ_GGUF_Q4_0 = 0,   /* 32 weights in 18 bytes: fp16 d, 16 bytes of nibbles; w = d * (nibble - 8) */
    UQ_GGUF_Q8_0 = 1    /* 32 weights in 34 bytes: fp16 d, 32 signed bytes q; w = d * q */
} uq_gguf_type;

/* Human-readable name of a status code (static string, never NULL). */
const char* uq_status_string(uq_status s);

/* Message of the last error raised on the calling thread (static per thread, never NULL). */
const char* uq_last_error(void);

/*
 * uq_packed_size -- bytes of every buffer a (N, K, group, fmt) weight needs.
 *   wq_bytes     packed code plane written by uq_pack_layout: Np*Kp*bits/8 with N padded
 *                to Np (a multiple of 16) and K to Kp (a multiple of 64 4-bit, 128 2-bit or
 *                32 8-bit codes), so at least N*K*bits/8
 *   scales_bytes `scales` argument of uq_gemm: fp16 [N][K/group]; UQ_K4: 16-byte
 *                records [N][K/256] written by uq_pack_kmeta
 *   zeros_bytes  `zeros_or_codebook` argument: UQ_INT4_ASYM uint8 [N][ceil(K/group/2)]
 *                (two 4-bit zeros per byte, low nibble = even group); UQ_INT2_ASYM fp16
 *                [N][K/group]; UQ_NF4 64 (fp32 c[16]); others 0 (pass NULL)
 * Host-only; any output pointer may be NULL.  Returns UQ_ERR_INVALID / UQ_ERR_UNSUPPORTED
 * under the same rules as uq_gemm.
 */
uq_status uq_packed_size(int N, int K, int group, uq_fmt fmt,
                         size_t* wq_bytes, size_t* scales_bytes, size_t* zeros_bytes);

/*
 * uq_pack_layout -- codes -> the kernels' packed code plane ("pack multiple low-bit
 * values into bytes", section "Quantization").
 *   codes (device)  int8 [N][K] row-major: the signed code for the SYM formats, the
 *                   unsigned code (stored in int8) otherwise.
 *   wq    (device)  uq_packed_size(...).wq_bytes bytes, written.
 * Layout (library-defined): rows in blocks of 16 (padding rows hold code 0), k in
 * chunks of 512 bytes per row block (32 lanes x 16 bytes), 16 chunks to an 8 KB tile;
 * the tiles of a row block follow in k order (the last one narrower when K is not a
 * multiple of the tile), row blocks follow each other.  Inside a chunk each 16-byte
 * lane slice holds the codes of rows g and g + 8 in the order of the mma.m16n8k16 A
 * fragment, so a shift and a lop3 per register unpack a bf16 pair.  Signed formats are
 * stored biased (+8, +128).  Offline call: it SYNCHRONIZES `stream`
 * and returns UQ_ERR_INVALID if any code is outside the format's range (wq is then
 * unspecified).
 */
uq_status uq_pack_layout(const int8_t* codes, void* wq, int N, int K, int group, uq_fmt fmt,
                         void* stream);

/*
 * uq_pack_gguf -- GGUF block-quantized weights -> the library's packed plane and scales ("Ultra LLM
 * Engine", section "Checkpoint Loading": GGUF block formats such as Q4_0; the other page's GGUF loader
 * dequantizes them).  Q4_0 is exactly UQ_INT4_SYM with group 32 (code = nibble - 8, scale = d) and Q8_0
 * exactly UQ_INT8_SYM with group 32 (code = q, scale = d), so the result feeds uq_gemm, uq_gemm_gated and
 * uq_dequant with that format and group 32, and decodes to the same W_hat as the blocks.
 *   blocks (device) the GGUF tensor's bytes: N rows of K/32 blocks (18 or 34 bytes each), byte aligned
 *   wq (device) uq_packed_size(N, K, 32, fmt).wq_bytes, written; scales (device) fp16 [N][K/32], written.
 * K a multiple of 32.  Asynchronous.
 */
uq_status uq_pack_gguf(const void* blocks, uq_gguf_type type, void* wq, uint16_t* scales, int N, int K, void* stream);

/*
 * uq_pack_kmeta -- UQ_K4 metadata -> 16-byte records [N][K/256] (the `scales` argument).
 *   d, dmin (device) fp16 [N][K/256];  sc, m (device) uint8 [N][K/256][8], values 0..63.
 *   meta    (device) 16*N*(K/256) bytes, written.  Record: fp16 d, fp16 dmin, then 8
 *           6-bit sc codes (bytes 4..9) and 8 6-bit m codes (bytes 10..15), little-endian
 *           bit order.  Offline call: synchronizes `stream`; UQ_ERR_INVALID if a code > 63.
 */
uq_status uq_pack_kmeta(const uint16_t* d, const uint16_t* dmin, const uint8_t* sc,
                        const uint8_t* m, void* meta, int N, int K, void* stream);

/*
 * uq_gemm -- y = x . W_hat^T with W_hat dequantized on the fly (the decode hot path).
 *   x      (device) bf16 [M][K] row-major
 *   wq     (device) packed codes from uq_pack_layout
 *   scales (device) fp16 [N][K/group] (s, or a for UQ_NF4); UQ_K4: records from uq_pack_kmeta
 *   zeros_or_codebook (device) see uq_packed_size; must be NULL for INT4_SYM, INT8_SYM, K4
 *   y      (device) bf16 [M][N] row-major, written (round to nearest even)
 *   M >= 0, N >= 0, K >= 0; M == 0 or N == 0 is a no-op; K == 0 writes zeros.
 *   group: 32, 64 or 128 for the flat formats (K % group == 0; UQ_INT2_ASYM also needs
 *   K % 64 == 0); 256 for UQ_K4 (K % 256 == 0).
 * Paths, per block of rows of x:
 *   - M <= 8: the GEMV on mma.sync (NF4's codebook values as two bf16 parts, hi + lo, with 16
 *     significant bits): one launch when each CTA owns whole row blocks, else the GEMV and a second
 *     launch that sums each row's partials in a fixed order, so repeated calls are bit-identical,
 *     and a row of x gives the same bits whatever the other rows of a call of M <= 8;
 *   - INT4_SYM, INT4_ASYM, INT2_ASYM with 9 <= M <= 15, and K4 with M >= 9: the mma.sync GEMM in
 *     blocks of 64 rows (each warp reuses an unpacked 16 x 16 block of exact integer (q - z) for
 *     every 8 columns of x; K4 adds a small column-sum launch, a k range split between CTAs a
 *     second pass), a last block of at most 8 rows on the GEMV;
 *   - every other M >= 16 with K a multiple of the code tile (1024 4-bit / 512 8-bit / 2048 2-bit
 *     codes): the tcgen05 tensor-core kernel in blocks of 64 rows; otherwise the GEMV over 8-row
 *     blocks.  uq_set_gemm_path can force either GEMM.
 * uq_gemm_kernel_count gives the launches of a shape.
 * Scratch: a library-owned workspace per (device, stream), grown on the first call
 * that needs more; that growth is refused (UQ_ERR_NOMEM) while `stream` is being
 * captured, so make one call of the largest size before capturing.  A buffer replaced
 * by growth is kept allocated until the process exits, so a CUDA graph captured before
 * the growth stays valid and may be replayed afterwards.  Calls on the same stream are
 * serialised by the stream; concurrent streams use separate workspaces.  A captured
 * graph uses the workspace of the stream it was captured on: do not run it concurrently
 * with other calls on that stream (or with another replay of itself).
 */
uq_status uq_gemm(const uint16_t* x, const void* wq, const void* scales,
                  const void* zeros_or_codebook, uint16_t* y,
                  int M, int N, int K, int group, uq_fmt fmt, void* stream);

/*
 * uq_gemm_gated -- the gated MLP's gate and up projections with the SiLU-multiply epilogue
 * ("Ultra LLM Engine", section "How the Engine Works": every layer ends in a gated MLP; read as the
 * Llama-style SiLU gate):
 *     h[m][n] = bf16_RNE( silu(g) * u ),  g = sum_k x[m][k] W_gate_hat[n][k],  u = sum_k x[m][k] W_up_hat[n][k],
 * g and u accumulated in fp32 exactly as uq_gemm does, silu(g) = g / (1 + e^-g) and the product in
 * fp32, one rounding to bf16 (no bf16 rounding of g or u).
 *   x (device) bf16 [M][K]; wq_gate / scales_gate / zc_gate and wq_up / scales_up / zc_up (device):
 *   two weights of the same N, K, group and format, each as uq_gemm takes them; h (device) bf16
 *   [M][N], written.  M == 0 or N == 0 is a no-op; K == 0 writes zeros.
 * Paths, routed as uq_gemm: every format with M <= 8 (and a last block of at most 8 rows after
 * mma.sync GEMM blocks) runs one mma-GEMV launch over both weights (gate
 * and up row blocks interleaved, each CTA owning whole gate/up pairs, h formed in its per-row
 * reduction), plus the second pass when the work split shares row blocks between CTAs; everything
 * else (the mma.sync GEMM, the tensor-core path) runs the gate projection into
 * fp32 library scratch and then the up projection, whose epilogue reads g and writes h.
 * uq_gemm_gated_kernel_count gives the launches.
 * Scratch, errors and stream capture as uq_gemm (the fp32 gate scratch, rows x N floats, is part of
 * the per-stream workspace).
 */
uq_status uq_gemm_gated(const uint16_t* x, const void* wq_gate, const void* scales_gate, const void* zc_gate,
                        const void* wq_up, const void* scales_up, const void* zc_up, uint16_t* h,
                        int M, int N, int K, int group, uq_fmt fmt, void* stream);

/* uq_gemm_gated_kernel_count -- kernels one uq_gemm_gated call of this shape launches (as uq_gemm_kernel_count). */
uq_status uq_gemm_gated_kernel_count(int M, int N, int K, int group, uq_fmt fmt, int* count);

/*
 * uq_rope_table -- the cos/sin table of rotary position embedding for uq_rmsnorm_rope:
 *     table[p][i] = ( cos(p * base^(-2i/head_dim)), sin(p * base^(-2i/head_dim)) ),  p < max_pos, i < head_dim/2,
 * evaluated in fp64 and rounded to fp32 (table: device, fp32 [max_pos][head_dim/2][2], written).
 * Build it once per (max_pos, head_dim, base).  head_dim even, base > 1.  Asynchronous.
 */
uq_status uq_rope_table(float* table, int max_pos, int head_dim, double base, void* stream);

/*
 * uq_rmsnorm_rope -- RMSNorm followed by rotary position embedding, fused ("Ultra LLM Engine", section
 * "Fused Kernels": RMSNorm followed by RoPE; read as the Llama-style RMSNorm and rotate-half RoPE):
 *     n[m][j] = x[m][j] / sqrt(mean_j(x[m][j]^2) + eps) * gamma[j]        (over the row's D values)
 *     every head_dim block of row m rotated by the row's position p = pos[m]: for i < head_dim/2,
 *     (n_i, n_{i+h/2}) -> (n_i cos - n_{i+h/2} sin, n_{i+h/2} cos + n_i sin), (cos, sin) = table[p][i]
 *     y[m][j] = bf16_RNE of the result (fp32 arithmetic throughout).
 *   x, y (device) bf16 [M][D] (y may be x); gamma (device) bf16 [D]; pos (device) int32 [M];
 *   table from uq_rope_table with the same head_dim; head_dim a multiple of 16; D a multiple of head_dim.
 * A row may be a token's hidden vector or one head's vector (per-head query/key norm: D = head_dim).
 * A position outside [0, max_pos) leaves its row unwritten and sets bit 3 of the fault word
 * (uq_device_fault).  Asynchronous.
 */
uq_status uq_rmsnorm_rope(const uint16_t* x, const uint16_t* gamma, const int32_t* pos, const float* table,
                          uint16_t* y, int M, int D, int head_dim, int max_pos, float eps, void* stream);

/*
 * uq_gemm_w4a8 -- the quantized linear layer with dynamically quantized activations ("Ultra LLM Engine",
 * section "Quantized Model": activations dynamically quantized for the GEMV/GEMM paths; read as
 * symmetric per-row int8):
 *     s_x[m] = absmax_k |x[m][k]| / 127 (fp32),  xq = clamp(RNE(x / s_x), -127, 127) (fp32 quotient),
 *     y[m][n] = bf16_RNE( s_x[m] * sum_g s[n][g] * sum_{k in g} xq[m][k] * (q[n][k] - z[n][g]) ),
 * the inner sums exact integers (integer tensor instructions, u8 x s8 -> s32), the per-group scaling
 * and the sum over groups in fp32.
 * Weights: UQ_INT4_SYM, UQ_INT4_ASYM (W4A8) or UQ_INT8_SYM (W8A8), as uq_gemm takes them.  Arguments,
 * layouts, errors and scratch as uq_gemm (the x codes, s_x and the per-group code sums live in the
 * per-stream workspace).  Launches: the activation quantization, then per block of 8 rows of x the
 * integer GEMV (plus its second pass when the work split shares row blocks between CTAs);
 * uq_gemm_w4a8_kernel_count gives the total.  The result differs from uq_gemm's by the activation
 * quantization: that is the method, not an error.
 */
uq_status uq_gemm_w4a8(const uint16_t* x, const void* wq, const void* scales, const void* zeros, uint16_t* y,
                       int M, int N, int K, int group, uq_fmt fmt, void* stream);

/* uq_gemm_w4a8_kernel_count -- kernels one uq_gemm_w4a8 call of this shape launches. */
uq_status uq_gemm_w4a8_kernel_count(int M, int N, int K, int group, uq_fmt fmt, int* count);

/*
 * uq_unpack_codes -- debug: packed plane -> int8 codes [N][K] (device), bit-exact
 * inverse of uq_pack_layout.  It decodes every code word with the register unpacking
 * the GEMV and tensor-core kernels run (shift + lop3 magic-exponent pairs for 4- and
 * 2-bit codes, the fp32 byte magic for 8-bit codes).
 */
uq_status uq_unpack_codes(const void* wq, int8_t* codes, int N, int K, int group, uq_fmt fmt,
                          void* stream);

/*
 * uq_dequant -- debug: W_hat as fp32 [N][K] (device), the correctly rounded value of the
 * format's reconstruction formula (bit-exact against an exact evaluation).
 */
uq_status uq_dequant(const void* wq, const void* scales, const void* zeros_or_codebook,
                     float* w, int N, int K, int group, uq_fmt fmt, void* stream);

/*
 * uq_quantize -- GPU quantizer for the flat formats (INT4_SYM, INT4_ASYM, INT8_SYM,
 * INT2_ASYM, NF4): fp32 W [N][K] (device) -> int8 codes [N][K], fp16 scales
 * [N][K/group], zeros (INT4_ASYM: uint8 [N][K/group], one zero per byte, NOT the
 * nibble-packed uq_gemm layout -- use uq_pack_zeros; INT2_ASYM: fp16 [N][K/group];
 * else NULL) and, for NF4, the input codebook fp32 c[16] (ascending).
 * Rules (scales in float64 then fp16): symmetric s = fp16_RNE(absmax/qmax),
 * q = clamp(rint(w/s)); asymmetric s = fp16 toward +inf of (max(w,0)-min(w,0))/L,
 * z = rint(-min/s), q = clamp(rint(w/s)+z, 0, L); NF4 a = fp16_RNE(absmax),
 * q = first index minimising |w/a - c[i]|.  Offline; asynchronous.
 */
uq_status uq_quantize(const float* w, int8_t* codes, uint16_t* scales, void* zeros,
                      const float* codebook, int N, int K, int group, uq_fmt fmt, void* stream);

/*
 * uq_quantize_k4 -- GPU quantizer for UQ_K4: fp32 W [N][K] -> codes int8 [N][K],
 * fp16 d, dmin [N][K/256], uint8 sc, m [N][K/256][8] (min/max quantizer with
 * ceilings: dmin = fp16 up of max(-lo_j)/63, m_j = ceil(-lo_j/dmin),
 * d = fp16 up of max(hi_j + dmin*m_j)/945, sc_j = ceil(r_j/(15d)),
 * q = clamp(rint((w + dmin*m_j)/(d*sc_j)), 0, 15)).  Offline; asynchronous.
 */
uq_status uq_quantize_k4(const float* w, int8_t* codes, uint16_t* d, uint16_t* dmin,
                         uint8_t* sc, uint8_t* m, int N, int K, void* stream);

/*
 * uq_pack_zeros -- INT4_ASYM zeros, one per byte [N][G] (device) -> the uq_gemm layout
 * [N][ceil(G/2)] (two per byte, low nibble = even group).  Asynchronous.
 */
uq_status uq_pack_zeros(const uint8_t* zeros, uint8_t* packed, int N, int G, void* stream);

/*
 * uq_set_gemm_path -- process-wide choice (default 0) of the GEMM for blocks of rows of x of the
 * 4-bit and 2-bit formats: 0 = automatic (as uq_gemm lists); 1 = the tcgen05 tensor-core kernel for
 * every block of 16..64 rows whose shape it supports; 2 = the mma.sync GEMM for every block of
 * 9..64 rows.  For comparing and testing the paths: all of them meet the same rule, but their
 * roundings differ, so they are not bit-identical to each other.  Host-only; UQ_ERR_INVALID for
 * another value.
 */
uq_status uq_set_gemm_path(int path);

/*
 * uq_set_launch_overlap -- process-wide switch (default 0 = off) for how uq_gemm launches its
 * GEMV and tensor-core kernels.  When on, each launch uses programmatic dependent launch: the kernel may
 * begin while the previous kernel on the same stream is still finishing, and streams its packed
 * weights, scales and zero points from HBM during that time; it waits for the previous kernel to
 * complete before it reads x, touches the split-K workspace or writes y.  Turn it on only when
 * wq / scales / zeros_or_codebook are not written by the work that immediately precedes the
 * call on the stream (true for a decode loop over fixed weights).  Host-only; always UQ_OK.
 */
uq_status uq_set_launch_overlap(int enable);

/*
 * uq_gemm_kernel_count -- how many kernels uq_gemm launches for this shape on the current device
 * (the GEMV and its second pass for rows shared between SMs; the mma.sync GEMM with its x
 * column sums (K4) and second pass; the tensor-core kernel with its x column sums (K4)), for
 * callers that account for launches.  Queries the device's SM count
 * (CUDA runtime, no kernel launched, nothing allocated).  *count = 0 for an empty call.
 * UQ_ERR_INVALID / UQ_ERR_UNSUPPORTED as uq_gemm for shapes it rejects.
 */
uq_status uq_gemm_kernel_count(int M, int N, int K, int group, uq_fmt fmt, int* count);

/*
 * uq_device_fault -- reads and clears the device-side fault words of the current device: the
 * one of uq_gemm and the one of uq_gemm_noalloc, OR-ed together (bit 0 / bit 1: a GEMV /
 * tensor-core kernel's bounded wait ran out and the kernel returned early instead of hanging;
 * its output is then unspecified; bit 2: a GEMV launch was given a work split larger than the
 * kernel holds and computed nothing; bit 3: uq_rmsnorm_rope met a position outside its table).  Synchronizes the device; allocates nothing.
 * *flag = 0 when no fault.
 */
uq_status uq_device_fault(unsigned int* flag);

/*
 * uq_gemm_noalloc -- uq_gemm's small-M GEMV for callers that cannot let a library allocate device
 * memory.  The reference pages have no counterpart: it exists for integration, not for the method.
 * Such callers include serving runtimes that reserve all device memory at start-up and forbid
 * later allocation (where cudaMalloc fails or steals memory promised elsewhere), and latency-
 * critical loops that cannot take the implicit device synchronisation of cudaMalloc/cudaFree.
 * Same arguments, layouts and result as uq_gemm (x, wq, scales, zeros_or_codebook, y are caller-
 * owned device buffers), computed with the same GEMV kernel for every M (row blocks of 8; no
 * GEMM path), so the output equals uq_gemm's for M <= 8.
 * Scratch: a 1 MiB static device array inside the library (every GPU that loads the library holds
 * it until the process exits); 256 bytes hold the fault word, and the rest must hold what the
 * launch's work split uses for one 8-row block of x (Mb = min(M, 8); uq_gemm_noalloc_scratch
 * reports it):
 *   nothing when every CTA owns whole 16-row blocks (the split uq_gemm_kernel_count reports as one
 *   launch); otherwise fp32 partial sums of every tile, 64*Mb*ceil(N/16)*ceil(K/T) bytes (T = 1024
 *   codes, 2048 for INT2_ASYM, 512 for INT8_SYM): ceil(N/16)*ceil(K/T)*Mb <= 16380.
 * Larger requests return UQ_ERR_NOMEM with the sizes in uq_last_error().  K == 0 returns
 * UQ_ERR_UNSUPPORTED.  Calls no cudaMalloc, cudaFree or other allocating routine.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  Every call shares the one
 * array and clears the part that must start at zero; calls whose kernels overlap on the GPU (for
 * example on two streams at once) race on it and must be serialised by the caller.  A wait that
 * runs out inside a no-alloc launch is reported by uq_device_fault like any other.
 */
uq_status uq_gemm_noalloc(const uint16_t* x, const void* wq, const void* scales,
                          const void* zeros_or_codebook, uint16_t* y,
                          int M, int N, int K, int group, uq_fmt fmt, void* stream);

/*
 * uq_gemm_noalloc_scratch -- the static scratch uq_gemm_noalloc would use for this shape on the
 * current device: *ticket_bytes (row-block tickets; 0: every GEMV sums its partials in a second
 * launch) and *partial_bytes (fp32 partial sums; 0 when every CTA owns whole row blocks), as listed
 * above.
 * Host-only (queries the SM count).  UQ_ERR_INVALID /
 * UQ_ERR_UNSUPPORTED as uq_gemm_noalloc for shapes it rejects; it does not check the 1 MiB limit.
 */
uq_status uq_gemm_noalloc_scratch(int M, int N, int K, int group, uq_fmt fmt, size_t* ticket_bytes,
                                  size_t* partial_bytes);

#ifdef __cplusplus
}
#endif

#endif /* UQ_H */
