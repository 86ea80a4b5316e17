// uq_gemv.cuh -- small-M (M <= 8) fused dequantize + GEMV/GEMM on CUDA cores, sm_103a.
//
// "Ultra LLM Engine", section "Fused Kernels": dequantized-weight GEMV for single-token
// decode and GEMM for batched decode.  Decode is bound by streaming the packed weights
// from HBM once, so the kernel is organised around that stream:
//
//  * Work is the list of tiles (8 rows x 512 bytes of codes) in row-block-major order.
//    Every warp is an independent worker that owns a contiguous, equal share of that list
//    (a "stream-K" split: perfectly balanced over 152 SMs x 8 warps whatever N and K are).
//  * Each warp keeps GEMV_STAGES tiles in flight: lane 0 issues one 1-D bulk async copy
//    (cp.async.bulk, completion counted in bytes on an mbarrier) per tile into a
//    warp-private ring in shared memory; there is no block-level synchronisation.
//  * Lane l owns the 16-byte column chunk l of every tile row (32 INT4 codes).  Its slice
//    of x stays in registers while it walks the 8 rows; codes are unpacked with the
//    magic-exponent trick (bf16 0x4300 | code = 128 + code) and multiplied-accumulated with
//    fma.rn.f32.bf16 (fp32 accumulate of exact bf16 products).  The +128 offset and the
//    zero point are removed once per group: sum x*(q - z) = sum x*(128 + q) - (128 + z)*sum x.
//  * Group scales are applied once per lane chunk (a chunk never spans two groups except
//    INT2 with group 32, handled as two halves).
//  * A row block whose k range is split between workers is finished by a deterministic
//    second pass: each contributor stores its fp32 partial sums, takes a ticket, and the
//    last one sums the partials in worker order (fixed, so results are bit-reproducible)
//    and writes y.  No worker ever waits for another.
#pragma once
#include "uq_kernels.h"

namespace uq {

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

// per-row metadata of the lane's chunk, converted to what the accumulate step needs
struct RowMeta {
    float s;     // scale (s, a, or d*sc for K4)
    float zc;    // value subtracted per unit of sum(x): 128 + z (INT*), 136 (INT4_SYM), 128 (K4)
    float s2;    // INT2 group-32 second half: scale;  K4: dmin*m
    float zc2;   // INT2 group-32 second half: 128 + z
};

template <int FMT>
__device__ __forceinline__ RowMeta load_meta(const GemvArgs& a, int n, int k0) {
    RowMeta r{0.f, 0.f, 0.f, 0.f};
    if constexpr (FMT == UQ_K4) {
        const int sb = k0 >> 8, j = (k0 & 255) >> 5;
        uint4 rec = ldg_nc_v4(a.scales + ((long long)n * (a.K >> 8) + sb) * 16);
        float d = half_bits_f32((uint16_t)(rec.x & 0xFFFF));
        float dmin = half_bits_f32((uint16_t)(rec.x >> 16));
        uint64_t sc48 = (uint64_t)rec.y | ((uint64_t)(rec.z & 0xFFFFu) << 32);
        uint64_t m48 = (uint64_t)(rec.z >> 16) | ((uint64_t)rec.w << 16);
        r.s = d * (float)((sc48 >> (6 * j)) & 63);
        r.s2 = dmin * (float)((m48 >> (6 * j)) & 63);
        r.zc = 128.0f;
    } else {
        const int G = a.K / a.group;
        const int gi = k0 / a.group;
        const uint16_t* sp = reinterpret_cast<const uint16_t*>(a.scales) + (long long)n * G;
        r.s = half_bits_f32(__ldg(sp + gi));
        if constexpr (FMT == UQ_INT4_SYM) {
            r.zc = 136.0f;
        } else if constexpr (FMT == UQ_INT4_ASYM) {
            const uint32_t b = __ldg(a.zc + (long long)n * ((G + 1) >> 1) + (gi >> 1));
            // fp32 with exponent 134 and z at mantissa bits 16..19 is exactly 128 + z
            r.zc = __uint_as_float(0x43000000u | (((gi & 1) ? (b >> 4) : (b & 15u)) << 16));
        } else if constexpr (FMT == UQ_INT2_ASYM) {
            const uint16_t* zp = reinterpret_cast<const uint16_t*>(a.zc) + (long long)n * G;
            r.zc = 128.0f + half_bits_f32(__ldg(zp + gi));
            if (a.group == 32) {
                r.s2 = half_bits_f32(__ldg(sp + gi + 1));
                r.zc2 = 128.0f + half_bits_f32(__ldg(zp + gi + 1));
            }
        }
    }
    return r;
}

// One pass over the tile's rows for x rows M0 .. M0+MP-1.  xg points at x[M0][k0].
template <int FMT, int M, int M0, int MP>
__device__ __forceinline__ void tile_pass(const uint8_t* __restrict__ tile, int slice_bytes, int rows,
                                          int lane, const uint16_t* __restrict__ xg, int ldx,
                                          const RowMeta (&meta)[RB], float (&acc)[RB][M],
                                          const float* __restrict__ lut, bool two_groups,
                                          const float* __restrict__ sxt) {
    constexpr int CPL = fmt_cpl(FMT);
    if constexpr (FMT == UQ_INT4_SYM || FMT == UQ_INT4_ASYM || FMT == UQ_K4 || FMT == UQ_INT2_ASYM) {
        // x as bf16 pairs: CPL/2 registers per row of x
        constexpr int XR = CPL / 2;
        uint32_t xr[MP][XR];
        float sx[MP], sx2[MP];
#pragma unroll
        for (int i = 0; i < MP; ++i) {
            const uint16_t* xp = xg + (long long)i * ldx;
#pragma unroll
            for (int v = 0; v < XR / 4; ++v) {
                uint4 q = ldg_nc_v4(xp + 8 * v);
                xr[i][4 * v] = q.x; xr[i][4 * v + 1] = q.y; xr[i][4 * v + 2] = q.z; xr[i][4 * v + 3] = q.w;
            }
            // sum of x over the lane's chunk (first / second half for INT2 with group 32),
            // precomputed per k tile into shared memory at kernel start
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
            const uint16_t* xp = xg + (long long)i * ldx;
#pragma unroll
            for (int v = 0; v < CPL / 8; ++v) {
                uint4 q = ldg_nc_v4(xp + 8 * v);
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

template <int FMT, int M, int M0>
__device__ __forceinline__ void tile_all_passes(const uint8_t* tile, int slice_bytes, int rows, int lane,
                                                const uint16_t* xg, int ldx, const RowMeta (&meta)[RB],
                                                float (&acc)[RB][M], const float* lut, bool two_groups,
                                                const float* sxt) {
    if constexpr (M0 < M) {
        constexpr int REM = M - M0;
        constexpr int MP = REM < PassPlan<FMT>::MAXP ? REM : PassPlan<FMT>::MAXP;
        tile_pass<FMT, M, M0, MP>(tile, slice_bytes, rows, lane, xg + (long long)M0 * ldx, ldx, meta, acc,
                                  lut, two_groups, sxt);
        tile_all_passes<FMT, M, M0 + MP>(tile, slice_bytes, rows, lane, xg, ldx, meta, acc, lut, two_groups, sxt);
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

template <int FMT, int M>
__global__ void __launch_bounds__(GEMV_WARPS * 32, 1) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int KT = fmt_kt(FMT), CPL = fmt_cpl(FMT);
    constexpr bool NEEDS_SX = (FMT != UQ_INT8_SYM && FMT != UQ_NF4);
    uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + GEMV_WARPS * GEMV_STAGES * TILE_BYTES);
    float* lut = reinterpret_cast<float*>(bars_all + GEMV_WARPS * GEMV_STAGES);
    // sx table [kb][h][m][lane]: sum of x[m] over lane chunk (half h of it for INT2 group 32)
    float* sx_tab = lut + 16;
    const int KBt = (a.K + KT - 1) / KT;
    constexpr int HALVES = (FMT == UQ_INT2_ASYM) ? 2 : 1;
    if constexpr (FMT == UQ_NF4) {
        if (threadIdx.x < 16) lut[threadIdx.x] = reinterpret_cast<const float*>(a.zc)[threadIdx.x];
    }
    if constexpr (NEEDS_SX) {
        const bool split = (FMT == UQ_INT2_ASYM) && (a.group == 32);
        for (int e = threadIdx.x; e < KBt * M * 32; e += blockDim.x) {
            const int kb = e / (M * 32), m = (e / 32) % M, l = e % 32;
            const int k0 = kb * KT + l * CPL;
            float s0 = 0.f, s1 = 0.f;
            if (k0 < a.K) {
                const uint16_t* xp = a.x + (long long)m * a.ldx + k0;
#pragma unroll
                for (int v = 0; v < CPL / 8; ++v) {
                    const uint4 q = ldg_nc_v4(xp + 8 * v);
                    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float t = bf16lo_f32(u[j]) + bf16hi_f32(u[j]);
                        if (4 * v + j < CPL / 4) s0 += t; else s1 += t;
                    }
                }
            }
            float* row = sx_tab + (long long)kb * HALVES * M * 32;
            if (split) {
                row[m * 32 + l] = s0;
                row[(M + m) * 32 + l] = s1;
            } else {
                row[m * 32 + l] = s0 + s1;
            }
        }
    }
    if constexpr (FMT == UQ_NF4 || NEEDS_SX) __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = blockIdx.x * GEMV_WARPS + warp;
    if (w >= a.P) return;

    const Layout L(a.N, a.K, FMT);
    uint8_t* ring = smem + warp * GEMV_STAGES * TILE_BYTES;
    uint64_t* bars = bars_all + warp * GEMV_STAGES;
    const long long t0 = range_begin(w, a.T, a.P), t1 = range_begin(w + 1, a.T, a.P);
    const int first_nb = (int)(t0 / L.KB);
    const bool two_groups = (FMT == UQ_INT2_ASYM) && (a.group == 32);

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < GEMV_STAGES; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
        fence_proxy_async_smem();
        for (int s = 0; s < GEMV_STAGES && t0 + s < t1; ++s) {
            const long long t = t0 + s;
            const int nb = (int)(t / L.KB), kb = (int)(t % L.KB);
            const uint32_t bytes = (uint32_t)(L.rows(nb) * L.slice_bytes(kb));
            mbar_arrive_expect_tx(&bars[s], bytes);
            bulk_g2s(ring + s * TILE_BYTES, a.wq + L.tile_offset(nb, kb), bytes, &bars[s]);
        }
    }
    __syncwarp();

    float acc[RB][M];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

    for (long long t = t0; t < t1; ++t) {
        const int it = (int)(t - t0);
        const int s = it % GEMV_STAGES;
        const uint32_t parity = (uint32_t)((it / GEMV_STAGES) & 1);
        const int nb = (int)(t / L.KB), kb = (int)(t % L.KB);
        const int rows = L.rows(nb);
        const int n0 = nb * RB;
        const int width = L.width(kb);
        const bool active = lane * CPL < width;
        const int k0 = kb * KT + lane * CPL;

        RowMeta meta[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            meta[r] = RowMeta{0.f, 0.f, 0.f, 0.f};
            if (active && r < rows) meta[r] = load_meta<FMT>(a, n0 + r, k0);
        }

        if (!mbar_wait_bounded(&bars[s], parity, a.fault, FAULT_GEMV_WAIT)) {
            // give the copies still in flight a bounded chance to land, then leave
            for (int j = 1; j < GEMV_STAGES && t + j < t1; ++j) {
                const int sj = (it + j) % GEMV_STAGES;
                mbar_wait_bounded(&bars[sj], (uint32_t)(((it + j) / GEMV_STAGES) & 1), a.fault, FAULT_GEMV_WAIT);
            }
            return;
        }
        if (active)
            tile_all_passes<FMT, M, 0>(ring + s * TILE_BYTES, L.slice_bytes(kb), rows, lane,
                                       a.x + k0, a.ldx, meta, acc, lut, two_groups,
                                       sx_tab + (long long)kb * HALVES * M * 32);
        __syncwarp();
        if (lane == 0 && t + GEMV_STAGES < t1) {
            fence_proxy_async_smem();
            const long long tn = t + GEMV_STAGES;
            const int nbn = (int)(tn / L.KB), kbn = (int)(tn % L.KB);
            const uint32_t bytes = (uint32_t)(L.rows(nbn) * L.slice_bytes(kbn));
            mbar_arrive_expect_tx(&bars[s], bytes);
            bulk_g2s(ring + s * TILE_BYTES, a.wq + L.tile_offset(nbn, kbn), bytes, &bars[s]);
        }

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

inline size_t gemv_smem_bytes_impl(int fmt, int K, int M) {
    const size_t kbt = (size_t)(K + fmt_kt(fmt) - 1) / fmt_kt(fmt);
    const size_t sx = (fmt == UQ_INT8_SYM || fmt == UQ_NF4) ? 0 : kbt * (fmt == UQ_INT2_ASYM ? 2 : 1) * M * 32 * 4;
    return (size_t)GEMV_WARPS * GEMV_STAGES * TILE_BYTES + (size_t)GEMV_WARPS * GEMV_STAGES * 8 + 64 + sx;
}
inline size_t gemv_partials_floats_impl(int P, int M) { return (size_t)2 * P * RB * M; }

namespace gemv_detail {
template <int FMT, int M>
cudaError_t launch_one(const GemvArgs& a, int grid, cudaStream_t st) {
    static bool configured[64] = {};   // the shared-memory opt-in, once per device
    const size_t smem = gemv_smem_bytes_impl(FMT, a.K, a.M);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gemv_kernel<FMT, M>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    gemv_kernel<FMT, M><<<grid, GEMV_WARPS * 32, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace gemv_detail

template <int FMT>
cudaError_t launch_gemv_fmt(const GemvArgs& a, int grid, cudaStream_t st) {
    switch (a.M) {
        case 1: return gemv_detail::launch_one<FMT, 1>(a, grid, st);
        case 2: return gemv_detail::launch_one<FMT, 2>(a, grid, st);
        case 3: return gemv_detail::launch_one<FMT, 3>(a, grid, st);
        case 4: return gemv_detail::launch_one<FMT, 4>(a, grid, st);
        case 5: return gemv_detail::launch_one<FMT, 5>(a, grid, st);
        case 6: return gemv_detail::launch_one<FMT, 6>(a, grid, st);
        case 7: return gemv_detail::launch_one<FMT, 7>(a, grid, st);
        case 8: return gemv_detail::launch_one<FMT, 8>(a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace uq
