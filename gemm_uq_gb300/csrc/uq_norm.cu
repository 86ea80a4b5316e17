// uq_norm.cu -- fused RMSNorm followed by rotary position embedding, and its cos/sin table.
//
// "Ultra LLM Engine", section "Fused Kernels": a fused "RMSNorm followed by RoPE" operation; section
// "How the Engine Works": each layer applies RMSNorm and rotary position embeddings before the
// quantized attention projections.  Per row m of D values:
//     n_j = x_j / sqrt(mean(x^2) + eps) * gamma_j,
// then every head_dim block of the row is rotated by the row's position p: value i and value
// i + head_dim/2 by the angle p * base^(-2i/head_dim) (the rotate-half pairing).  A row may be a
// token's hidden vector or one head's vector (per-head query/key norm): the definition is the same.
//
// Memory-bound: each row is read twice (the second read hits L1/L2) and written once; cos/sin come
// from a table [max_pos][head_dim/2] of fp32 pairs built once in fp64 (uq_rope_table).
#include "uq_kernels.h"

namespace uq {

namespace {

// table[p][i] = (cos, sin)(p * base^(-2i/head_dim)), evaluated in fp64 and rounded to fp32
__global__ void rope_table_kernel(float2* __restrict__ table, int max_pos, int half, double log_base, int head_dim) {
    const long long total = (long long)max_pos * half;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int p = (int)(e / half), i = (int)(e % half);
        const double inv = exp(-2.0 * (double)i / (double)head_dim * log_base);
        double sn, cs;
        sincos((double)p * inv, &sn, &cs);
        table[e] = make_float2((float)cs, (float)sn);
    }
}

__device__ __forceinline__ float bf16_f(uint32_t w, int hi) { return hi ? bf16hi_f32(w) : bf16lo_f32(w); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// One CTA per row (grid-stride over rows); y may be x (each value is read and written by one thread,
// reads first).  Work unit = 8 rotation pairs: values [i0, i0 + 8) and
// [i0 + h/2, i0 + h/2 + 8) of one head, two 16-byte loads.  Pass 1 sums the squares (fp32, then a
// fixed-order warp and block reduction); pass 2 normalises, rotates and stores.
__global__ void __launch_bounds__(256) rmsnorm_rope_kernel(const uint16_t* x, const uint16_t* __restrict__ gamma,
                                                           const int32_t* __restrict__ pos, const float2* __restrict__ table,
                                                           uint16_t* y, int M, int D, int head_dim, int max_pos, float eps,
                                                           unsigned int* fault) {
    __shared__ float red[8];
    __shared__ float r_row;
    const int half = head_dim >> 1, upt = half >> 3;           // units per head
    const int units = D >> 4;                                  // 8 pairs = 16 values per unit
    for (int m = blockIdx.x; m < M; m += gridDim.x) {
        const uint16_t* xr = x + (long long)m * D;
        float ss = 0.f;
        for (int t = threadIdx.x; t < units; t += blockDim.x) {
            const int h = t / upt, i0 = (t % upt) * 8;
            const uint4 a = *reinterpret_cast<const uint4*>(xr + h * head_dim + i0);
            const uint4 b = *reinterpret_cast<const uint4*>(xr + h * head_dim + half + i0);
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float v0 = bf16lo_f32(w[j]), v1 = bf16hi_f32(w[j]);
                ss = fmaf(v0, v0, ss);
                ss = fmaf(v1, v1, ss);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.f;
            for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
            r_row = rsqrtf(tot / (float)D + eps);
        }
        __syncthreads();
        const float r = r_row;
        const int p = pos[m];
        if (p < 0 || p >= max_pos) {
            if (threadIdx.x == 0) atomicOr(fault, FAULT_ROPE_POS);
            __syncthreads();
            continue;
        }
        const float2* trow = table + (long long)p * half;
        uint16_t* yr = y + (long long)m * D;
        for (int t = threadIdx.x; t < units; t += blockDim.x) {
            const int h = t / upt, i0 = (t % upt) * 8;
            const int lo_off = h * head_dim + i0, hi_off = lo_off + half;
            const uint4 a = *reinterpret_cast<const uint4*>(xr + lo_off);
            const uint4 b = *reinterpret_cast<const uint4*>(xr + hi_off);
            const uint4 ga = *reinterpret_cast<const uint4*>(gamma + lo_off);
            const uint4 gb = *reinterpret_cast<const uint4*>(gamma + hi_off);
            const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
            const uint32_t gwa[4] = {ga.x, ga.y, ga.z, ga.w}, gwb[4] = {gb.x, gb.y, gb.z, gb.w};
            uint32_t oa[4], ob[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float ylo[2], yhi[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float2 cs = trow[i0 + 2 * j + e];
                    const float nl = bf16_f(wa[j], e) * r * bf16_f(gwa[j], e);
                    const float nh = bf16_f(wb[j], e) * r * bf16_f(gwb[j], e);
                    ylo[e] = fmaf(nl, cs.x, -nh * cs.y);
                    yhi[e] = fmaf(nh, cs.x, nl * cs.y);
                }
                oa[j] = pack_bf16(ylo[0], ylo[1]);
                ob[j] = pack_bf16(yhi[0], yhi[1]);
            }
            *reinterpret_cast<uint4*>(yr + lo_off) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
            *reinterpret_cast<uint4*>(yr + hi_off) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        }
        __syncthreads();                                       // red / r_row are reused by the next row
    }
}

}  // namespace

cudaError_t launch_rope_table(float* table, int max_pos, int head_dim, double base, cudaStream_t st) {
    const long long total = (long long)max_pos * (head_dim / 2);
    long long g = (total + 255) / 256;
    if (g > 65536) g = 65536;
    rope_table_kernel<<<(int)(g < 1 ? 1 : g), 256, 0, st>>>(reinterpret_cast<float2*>(table), max_pos, head_dim / 2,
                                                            log(base), head_dim);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm_rope(const uint16_t* x, const uint16_t* gamma, const int32_t* pos, const float* table,
                                uint16_t* y, int M, int D, int head_dim, int max_pos, float eps, unsigned int* fault,
                                int sms, cudaStream_t st) {
    const int grid = M < 8 * sms ? M : 8 * sms;
    rmsnorm_rope_kernel<<<grid, 256, 0, st>>>(x, gamma, pos, reinterpret_cast<const float2*>(table), y, M, D, head_dim,
                                              max_pos, eps, fault);
    return cudaGetLastError();
}

}  // namespace uq
