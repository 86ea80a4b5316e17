// uq_pack.cu -- offline kernels: pack codes / K4 metadata, the debug unpack and dequant exports,
// and the GPU quantizers.  "Ultra LLM Engine", section "Quantization": the quantizers pack low-bit
// values into bytes and expose matching dequantization helpers for the fused kernels.
#include "uq_kernels.h"

namespace uq {

// ----------------------------------------------------------------------------------------------
// pack / unpack / dequant: one thread per 32-bit word of the packed plane; each code slot of the
// word is mapped to its (row, k) by Layout::slot_nk.  Slots outside [N) x [K) are padding and
// hold the stored form of code 0.

// values (code + bias, as stored) of every slot of word w, through the register unpacking the GEMV
// and tensor-core kernels run on their code words: the shift + lop3 magic-exponent pairs
// (nib_pair_lop3 / crumb_pair_lop3: bf16 128 + code) and the fp32 byte magic for 8-bit codes
template <int P>
__device__ __forceinline__ void pair_codes(uint32_t t, int* v) {
    v[2 * P] = (int)bf16lo_f32(t) - 128;
    v[2 * P + 1] = (int)bf16hi_f32(t) - 128;
}
template <int FMT>
__device__ __forceinline__ void stored_codes(uint32_t w, int (&v)[fmt_cpw(FMT)]) {
    if constexpr (FMT == UQ_INT8_SYM) {
#pragma unroll
        for (int s = 0; s < 4; ++s) v[s] = (int)(byte_magic_f32(w, s) - 8388608.0f);
    } else if constexpr (FMT == UQ_INT2_ASYM) {
        pair_codes<0>(crumb_pair_lop3<0>(w), v); pair_codes<1>(crumb_pair_lop3<1>(w), v);
        pair_codes<2>(crumb_pair_lop3<2>(w), v); pair_codes<3>(crumb_pair_lop3<3>(w), v);
        pair_codes<4>(crumb_pair_lop3<4>(w), v); pair_codes<5>(crumb_pair_lop3<5>(w), v);
        pair_codes<6>(crumb_pair_lop3<6>(w), v); pair_codes<7>(crumb_pair_lop3<7>(w), v);
    } else {
        pair_codes<0>(nib_pair_lop3<0>(w), v); pair_codes<1>(nib_pair_lop3<1>(w), v);
        pair_codes<2>(nib_pair_lop3<2>(w), v); pair_codes<3>(nib_pair_lop3<3>(w), v);
    }
}

template <int FMT>
__global__ void pack_kernel(const int8_t* __restrict__ codes, uint8_t* __restrict__ wq, int N, int K,
                            unsigned int* __restrict__ bad) {
    constexpr int BITS = fmt_bits(FMT), CPW = fmt_cpw(FMT), BIAS = fmt_bias(FMT);
    constexpr int LO = (FMT == UQ_INT4_SYM) ? -8 : (FMT == UQ_INT8_SYM ? -128 : 0);
    constexpr int HI = (FMT == UQ_INT4_SYM) ? 7 : (FMT == UQ_INT8_SYM ? 127 : (FMT == UQ_INT2_ASYM ? 3 : 15));
    const Layout L(N, K, FMT);
    const long long words = L.bytes() / 4;
    for (long long wi = blockIdx.x * (long long)blockDim.x + threadIdx.x; wi < words;
         wi += (long long)gridDim.x * blockDim.x) {
        uint32_t word = 0;
        bool ok = true;
#pragma unroll
        for (int s = 0; s < CPW; ++s) {
            int n, k;
            L.slot_nk(wi * 4, s, &n, &k);
            int c = 0;
            if (n < N && k < K) {
                c = codes[(long long)n * K + k];
                ok &= (c >= LO) && (c <= HI);
            }
            const uint32_t u = (uint32_t)(c + BIAS) & ((1u << BITS) - 1u);
            word |= u << slot_bitpos(BITS, s);
        }
        if (!ok) atomicAdd(bad, 1u);
        reinterpret_cast<uint32_t*>(wq)[wi] = word;
    }
}

// GGUF blocks -> the packed plane: Q4_0 is INT4_SYM at group 32 (code = nibble - 8), Q8_0 is INT8_SYM at
// group 32 (code = signed byte).  A row of K weights is K / 32 blocks of BB bytes: fp16 d, then the codes
// (Q4_0: byte j holds weight j in its low nibble and weight j + 16 in its high nibble).
template <int FMT>
__global__ void pack_gguf_kernel(const uint8_t* __restrict__ blocks, uint8_t* __restrict__ wq, int N, int K) {
    constexpr int BITS = fmt_bits(FMT), CPW = fmt_cpw(FMT), BIAS = fmt_bias(FMT);
    constexpr int BB = (FMT == UQ_INT4_SYM) ? 18 : 34;
    const Layout L(N, K, FMT);
    const long long words = L.bytes() / 4;
    const int nb = K / 32;
    for (long long wi = blockIdx.x * (long long)blockDim.x + threadIdx.x; wi < words;
         wi += (long long)gridDim.x * blockDim.x) {
        uint32_t word = 0;
#pragma unroll
        for (int s = 0; s < CPW; ++s) {
            int n, k;
            L.slot_nk(wi * 4, s, &n, &k);
            int c = 0;
            if (n < N && k < K) {
                const uint8_t* blk = blocks + ((long long)n * nb + k / 32) * BB + 2;
                const int j = k & 31;
                if constexpr (FMT == UQ_INT4_SYM) c = ((j < 16 ? blk[j] : (blk[j - 16] >> 4)) & 15) - 8;
                else c = (int)(int8_t)blk[j];
            }
            word |= ((uint32_t)(c + BIAS) & ((1u << BITS) - 1u)) << slot_bitpos(BITS, s);
        }
        reinterpret_cast<uint32_t*>(wq)[wi] = word;
    }
}

// the blocks' fp16 d as the fp16 scales [N][K/32] of the group-32 format
__global__ void gguf_scales_kernel(const uint8_t* __restrict__ blocks, uint16_t* __restrict__ scales, long long nblk,
                                   int BB) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nblk; i += (long long)gridDim.x * blockDim.x)
        scales[i] = (uint16_t)(blocks[i * BB] | (blocks[i * BB + 1] << 8));
}

template <int FMT>
__global__ void unpack_kernel(const uint8_t* __restrict__ wq, int8_t* __restrict__ codes, int N, int K) {
    constexpr int CPW = fmt_cpw(FMT), BIAS = fmt_bias(FMT);
    const Layout L(N, K, FMT);
    const long long words = L.bytes() / 4;
    for (long long wi = blockIdx.x * (long long)blockDim.x + threadIdx.x; wi < words;
         wi += (long long)gridDim.x * blockDim.x) {
        const uint32_t word = reinterpret_cast<const uint32_t*>(wq)[wi];
        int v[CPW];
        stored_codes<FMT>(word, v);
#pragma unroll
        for (int s = 0; s < CPW; ++s) {
            int n, k;
            L.slot_nk(wi * 4, s, &n, &k);
            if (n < N && k < K) codes[(long long)n * K + k] = (int8_t)(v[s] - BIAS);
        }
    }
}

// dequant: W_hat in fp32, the correctly rounded value of the format's formula
template <int FMT>
__global__ void dequant_kernel(const uint8_t* __restrict__ wq, const uint8_t* __restrict__ scales,
                               const uint8_t* __restrict__ zc, float* __restrict__ w, int N, int K,
                               int group) {
    constexpr int CPW = fmt_cpw(FMT), BIAS = fmt_bias(FMT);
    const Layout L(N, K, FMT);
    const long long words = L.bytes() / 4;
    const int G = K / group;
    for (long long wi = blockIdx.x * (long long)blockDim.x + threadIdx.x; wi < words;
         wi += (long long)gridDim.x * blockDim.x) {
        const uint32_t word = reinterpret_cast<const uint32_t*>(wq)[wi];
        int v[CPW];
        stored_codes<FMT>(word, v);
#pragma unroll
        for (int s = 0; s < CPW; ++s) {
            int n, k;
            L.slot_nk(wi * 4, s, &n, &k);
            if (n >= N || k >= K) continue;
            const float q = (float)(v[s] - BIAS);
            float out;
            if constexpr (FMT == UQ_K4) {
                const int sb = k / 256, j = (k % 256) / 32;
                const uint4 rec = *reinterpret_cast<const uint4*>(scales + ((long long)n * (K / 256) + sb) * 16);
                const float d = half_bits_f32((uint16_t)(rec.x & 0xFFFF));
                const float dmin = half_bits_f32((uint16_t)(rec.x >> 16));
                const uint64_t sc48 = (uint64_t)rec.y | ((uint64_t)(rec.z & 0xFFFFu) << 32);
                const uint64_t m48 = (uint64_t)(rec.z >> 16) | ((uint64_t)rec.w << 16);
                const float dsc = d * (float)((sc48 >> (6 * j)) & 63);          // exact: 11 x 6 bits
                const float dmm = dmin * (float)((m48 >> (6 * j)) & 63);        // exact
                out = fmaf(dsc, q, -dmm);                                      // one rounding
            } else {
                const int gi = k / group;
                const float sv = half_bits_f32(reinterpret_cast<const uint16_t*>(scales)[(long long)n * G + gi]);
                if constexpr (FMT == UQ_NF4) {
                    out = __fmul_rn(sv, __ldg(reinterpret_cast<const float*>(zc) + (int)q));
                } else {
                    float z = 0.0f;
                    if constexpr (FMT == UQ_INT4_ASYM) {
                        const uint8_t b = zc[(long long)n * ((G + 1) / 2) + gi / 2];
                        z = (float)((gi & 1) ? (b >> 4) : (b & 15));
                    } else if constexpr (FMT == UQ_INT2_ASYM) {
                        z = half_bits_f32(reinterpret_cast<const uint16_t*>(zc)[(long long)n * G + gi]);
                    }
                    out = __fmul_rn(sv, q - z);
                }
            }
            w[(long long)n * K + k] = out;
        }
    }
}

// K4 metadata records: one thread per (row, super-block)
__global__ void pack_kmeta_kernel(const uint16_t* __restrict__ d, const uint16_t* __restrict__ dmin,
                                  const uint8_t* __restrict__ sc, const uint8_t* __restrict__ m,
                                  uint8_t* __restrict__ meta, long long count, unsigned int* bad) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < count;
         i += (long long)gridDim.x * blockDim.x) {
        uint64_t s48 = 0, m48 = 0;
        bool ok = true;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t a = sc[i * 8 + j], b = m[i * 8 + j];
            ok &= (a < 64) && (b < 64);
            s48 |= (uint64_t)(a & 63) << (6 * j);
            m48 |= (uint64_t)(b & 63) << (6 * j);
        }
        if (!ok) atomicAdd(bad, 1u);
        uint4 rec;
        rec.x = (uint32_t)d[i] | ((uint32_t)dmin[i] << 16);
        rec.y = (uint32_t)s48;
        rec.z = (uint32_t)(s48 >> 32) | ((uint32_t)m48 << 16);
        rec.w = (uint32_t)(m48 >> 16);
        *reinterpret_cast<uint4*>(meta + i * 16) = rec;
    }
}

__global__ void pack_zeros_kernel(const uint8_t* __restrict__ z, uint8_t* __restrict__ out, int N, int G) {
    const int ZB = (G + 1) / 2;
    const long long total = (long long)N * ZB;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        int n = (int)(i / ZB), j = (int)(i % ZB);
        uint8_t lo = z[(long long)n * G + 2 * j] & 15;
        uint8_t hi = (2 * j + 1 < G) ? (z[(long long)n * G + 2 * j + 1] & 15) : 0;
        out[i] = (uint8_t)(lo | (hi << 4));
    }
}

// ----------------------------------------------------------------------------------------------
// Quantizers (float64 arithmetic, the same operations in the same order as the CPU definitions)

// smallest fp16 >= v (v finite, >= 0)
__device__ __forceinline__ uint16_t f16_up_bits(double v) {
    uint16_t h = __half_as_ushort(__double2half(v));
    if ((double)__half2float(__ushort_as_half(h)) < v) h = (uint16_t)(h + 1);
    return h;
}
__device__ __forceinline__ double hval(uint16_t h) { return (double)__half2float(__ushort_as_half(h)); }

__device__ __forceinline__ double warp_max(double v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ double warp_min(double v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmin(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// one warp per (row, group); group <= 128 so each lane holds at most 4 weights
template <int FMT>
__global__ void quantize_kernel(const float* __restrict__ w, int8_t* __restrict__ codes,
                                uint16_t* __restrict__ scales, void* __restrict__ zeros,
                                const float* __restrict__ codebook, int N, int K, int group) {
    const int lane = threadIdx.x & 31;
    const long long G = K / group;
    const long long gid = blockIdx.x * (long long)(blockDim.x / 32) + (threadIdx.x / 32);
    if (gid >= (long long)N * G) return;
    const int per = group / 32;
    const long long base = (gid / G) * K + (gid % G) * group;
    double v[4];
    double amax = 0.0, lo = 0.0, hi = 0.0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] = 0.0;
        if (i < per) {
            v[i] = (double)w[base + i * 32 + lane];
            amax = fmax(amax, fabs(v[i]));
            lo = fmin(lo, v[i]);
            hi = fmax(hi, v[i]);
        }
    }
    int8_t* out = codes + base;
    if constexpr (FMT == UQ_INT4_SYM || FMT == UQ_INT8_SYM) {
        constexpr double QMAX = (FMT == UQ_INT4_SYM) ? 7.0 : 127.0;
        constexpr double QMIN = (FMT == UQ_INT4_SYM) ? -8.0 : -127.0;
        amax = warp_max(amax);
        uint16_t sb = __half_as_ushort(__double2half(amax / QMAX));
        double s = hval(sb);
        for (int i = 0; i < per; ++i) {
            double q = s > 0.0 ? rint(v[i] / s) : 0.0;
            out[i * 32 + lane] = (int8_t)fmin(fmax(q, QMIN), QMAX);
        }
        if (lane == 0) scales[gid] = sb;
    } else if constexpr (FMT == UQ_INT4_ASYM || FMT == UQ_INT2_ASYM) {
        constexpr double LV = (FMT == UQ_INT4_ASYM) ? 15.0 : 3.0;
        lo = warp_min(lo);
        hi = warp_max(hi);
        double span = hi - lo;
        uint16_t sb = f16_up_bits(span / LV);
        if (hval(sb) * LV < span) sb = (uint16_t)(sb + 1);
        double s = hval(sb);
        double z = s > 0.0 ? rint(-lo / s) : 0.0;
        for (int i = 0; i < per; ++i) {
            double q = s > 0.0 ? fmin(fmax(rint(v[i] / s) + z, 0.0), LV) : 0.0;
            out[i * 32 + lane] = (int8_t)q;
        }
        if (lane == 0) {
            scales[gid] = sb;
            if constexpr (FMT == UQ_INT4_ASYM) reinterpret_cast<uint8_t*>(zeros)[gid] = (uint8_t)z;
            else reinterpret_cast<uint16_t*>(zeros)[gid] = __half_as_ushort(__double2half(z));
        }
    } else {  // NF4
        amax = warp_max(amax);
        uint16_t ab = __half_as_ushort(__double2half(amax));
        double a = hval(ab);
        int zidx = 0;
        double zbest = fabs((double)codebook[0]);
        for (int c = 1; c < 16; ++c) {
            double t = fabs((double)codebook[c]);
            if (t < zbest) { zbest = t; zidx = c; }
        }
        for (int i = 0; i < per; ++i) {
            int best = zidx;
            if (a > 0.0) {
                double r = v[i] / a;
                double bd = fabs(r - (double)codebook[0]);
                best = 0;
                for (int c = 1; c < 16; ++c) {
                    double dd = fabs(r - (double)codebook[c]);
                    if (dd < bd) { bd = dd; best = c; }
                }
            }
            out[i * 32 + lane] = (int8_t)best;
        }
        if (lane == 0) scales[gid] = ab;
    }
}

// K4: one warp per (row, super-block); lane l holds weights 8l .. 8l+7 (sub-block l / 4)
__global__ void quantize_k4_kernel(const float* __restrict__ w, int8_t* __restrict__ codes,
                                   uint16_t* __restrict__ dout, uint16_t* __restrict__ dminout,
                                   uint8_t* __restrict__ scout, uint8_t* __restrict__ mout, int N, int K) {
    const int lane = threadIdx.x & 31;
    const long long S = K / 256;
    const long long sid = blockIdx.x * (long long)(blockDim.x / 32) + (threadIdx.x / 32);
    if (sid >= (long long)N * S) return;
    const long long base = (sid / S) * K + (sid % S) * 256 + lane * 8;
    double v[8];
    double lo = 0.0, hi = 0.0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = (double)w[base + i];
        lo = fmin(lo, v[i]);
        hi = fmax(hi, v[i]);
    }
    // sub-block extremes: reduce over the 4 lanes of a sub-block
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        lo = fmin(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmax(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    double neg = -lo;
    double negmax = warp_max(neg);
    uint16_t dminb = f16_up_bits(negmax / 63.0);
    if (hval(dminb) * 63.0 < negmax) dminb = (uint16_t)(dminb + 1);
    double dmin = hval(dminb);
    double m = dmin > 0.0 ? ceil(neg / dmin) : 0.0;
    if (m * dmin < neg) m += 1.0;
    double off = dmin * m;
    double r = hi + off;
    double R = warp_max(r);
    uint16_t db = f16_up_bits(R / 945.0);
    if (hval(db) * 945.0 < R) db = (uint16_t)(db + 1);
    double d = hval(db);
    double unit = 15.0 * d;
    double sc = unit > 0.0 ? ceil(r / unit) : 0.0;
    if (unit * sc < r) sc += 1.0;
    double ds = d * sc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        double q = ds > 0.0 ? fmin(fmax(rint((v[i] + off) / ds), 0.0), 15.0) : 0.0;
        codes[base + i] = (int8_t)q;
    }
    if ((lane & 3) == 0) {
        scout[sid * 8 + lane / 4] = (uint8_t)sc;
        mout[sid * 8 + lane / 4] = (uint8_t)m;
    }
    if (lane == 0) {
        dout[sid] = db;
        dminout[sid] = dminb;
    }
}

// ----------------------------------------------------------------------------------------------
// launchers

static int grid_for(long long work, int block) {
    long long g = (work + block - 1) / block;
    if (g > 65535LL * 16) g = 65535LL * 16;
    return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_pack(int fmt, const int8_t* codes, uint8_t* wq, int N, int K, unsigned int* bad,
                        cudaStream_t st) {
    long long words = Layout(N, K, fmt).bytes() / 4;
    int g = grid_for(words, 256);
    switch (fmt) {
        case UQ_INT4_SYM: pack_kernel<UQ_INT4_SYM><<<g, 256, 0, st>>>(codes, wq, N, K, bad); break;
        case UQ_INT4_ASYM: pack_kernel<UQ_INT4_ASYM><<<g, 256, 0, st>>>(codes, wq, N, K, bad); break;
        case UQ_INT8_SYM: pack_kernel<UQ_INT8_SYM><<<g, 256, 0, st>>>(codes, wq, N, K, bad); break;
        case UQ_INT2_ASYM: pack_kernel<UQ_INT2_ASYM><<<g, 256, 0, st>>>(codes, wq, N, K, bad); break;
        case UQ_NF4: pack_kernel<UQ_NF4><<<g, 256, 0, st>>>(codes, wq, N, K, bad); break;
        case UQ_K4: pack_kernel<UQ_K4><<<g, 256, 0, st>>>(codes, wq, N, K, bad); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_pack_gguf(int qtype, const uint8_t* blocks, uint8_t* wq, uint16_t* scales, int N, int K,
                             cudaStream_t st) {
    const int fmt = qtype == 0 ? UQ_INT4_SYM : UQ_INT8_SYM;
    const Layout L(N, K, fmt);
    const long long words = L.bytes() / 4;
    long long g = (words + 255) / 256;
    if (g > 65536) g = 65536;
    if (fmt == UQ_INT4_SYM) pack_gguf_kernel<UQ_INT4_SYM><<<(int)(g < 1 ? 1 : g), 256, 0, st>>>(blocks, wq, N, K);
    else pack_gguf_kernel<UQ_INT8_SYM><<<(int)(g < 1 ? 1 : g), 256, 0, st>>>(blocks, wq, N, K);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long nblk = (long long)N * (K / 32);
    long long g2 = (nblk + 255) / 256;
    if (g2 > 65536) g2 = 65536;
    gguf_scales_kernel<<<(int)(g2 < 1 ? 1 : g2), 256, 0, st>>>(blocks, scales, nblk, qtype == 0 ? 18 : 34);
    return cudaGetLastError();
}

cudaError_t launch_unpack(int fmt, const uint8_t* wq, int8_t* codes, int N, int K, cudaStream_t st) {
    long long words = Layout(N, K, fmt).bytes() / 4;
    int g = grid_for(words, 256);
    switch (fmt) {
        case UQ_INT4_SYM: unpack_kernel<UQ_INT4_SYM><<<g, 256, 0, st>>>(wq, codes, N, K); break;
        case UQ_INT4_ASYM: unpack_kernel<UQ_INT4_ASYM><<<g, 256, 0, st>>>(wq, codes, N, K); break;
        case UQ_INT8_SYM: unpack_kernel<UQ_INT8_SYM><<<g, 256, 0, st>>>(wq, codes, N, K); break;
        case UQ_INT2_ASYM: unpack_kernel<UQ_INT2_ASYM><<<g, 256, 0, st>>>(wq, codes, N, K); break;
        case UQ_NF4: unpack_kernel<UQ_NF4><<<g, 256, 0, st>>>(wq, codes, N, K); break;
        case UQ_K4: unpack_kernel<UQ_K4><<<g, 256, 0, st>>>(wq, codes, N, K); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_dequant(int fmt, const uint8_t* wq, const uint8_t* scales, const uint8_t* zc, float* w,
                           int N, int K, int group, cudaStream_t st) {
    long long words = Layout(N, K, fmt).bytes() / 4;
    int g = grid_for(words, 256);
    switch (fmt) {
        case UQ_INT4_SYM: dequant_kernel<UQ_INT4_SYM><<<g, 256, 0, st>>>(wq, scales, zc, w, N, K, group); break;
        case UQ_INT4_ASYM: dequant_kernel<UQ_INT4_ASYM><<<g, 256, 0, st>>>(wq, scales, zc, w, N, K, group); break;
        case UQ_INT8_SYM: dequant_kernel<UQ_INT8_SYM><<<g, 256, 0, st>>>(wq, scales, zc, w, N, K, group); break;
        case UQ_INT2_ASYM: dequant_kernel<UQ_INT2_ASYM><<<g, 256, 0, st>>>(wq, scales, zc, w, N, K, group); break;
        case UQ_NF4: dequant_kernel<UQ_NF4><<<g, 256, 0, st>>>(wq, scales, zc, w, N, K, group); break;
        case UQ_K4: dequant_kernel<UQ_K4><<<g, 256, 0, st>>>(wq, scales, zc, w, N, K, group); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_pack_kmeta(const uint16_t* d, const uint16_t* dmin, const uint8_t* sc, const uint8_t* m,
                              uint8_t* meta, long long count, unsigned int* bad, cudaStream_t st) {
    pack_kmeta_kernel<<<grid_for(count, 256), 256, 0, st>>>(d, dmin, sc, m, meta, count, bad);
    return cudaGetLastError();
}

cudaError_t launch_pack_zeros(const uint8_t* z, uint8_t* out, int N, int G, cudaStream_t st) {
    pack_zeros_kernel<<<grid_for((long long)N * ((G + 1) / 2), 256), 256, 0, st>>>(z, out, N, G);
    return cudaGetLastError();
}

cudaError_t launch_quantize(int fmt, const float* w, int8_t* codes, uint16_t* scales, void* zeros,
                            const float* codebook, int N, int K, int group, cudaStream_t st) {
    long long groups = (long long)N * (K / group);
    long long blocks = (groups + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    dim3 g((unsigned)blocks);
    switch (fmt) {
        case UQ_INT4_SYM: quantize_kernel<UQ_INT4_SYM><<<g, 256, 0, st>>>(w, codes, scales, zeros, codebook, N, K, group); break;
        case UQ_INT4_ASYM: quantize_kernel<UQ_INT4_ASYM><<<g, 256, 0, st>>>(w, codes, scales, zeros, codebook, N, K, group); break;
        case UQ_INT8_SYM: quantize_kernel<UQ_INT8_SYM><<<g, 256, 0, st>>>(w, codes, scales, zeros, codebook, N, K, group); break;
        case UQ_INT2_ASYM: quantize_kernel<UQ_INT2_ASYM><<<g, 256, 0, st>>>(w, codes, scales, zeros, codebook, N, K, group); break;
        case UQ_NF4: quantize_kernel<UQ_NF4><<<g, 256, 0, st>>>(w, codes, scales, zeros, codebook, N, K, group); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_quantize_k4(const float* w, int8_t* codes, uint16_t* d, uint16_t* dmin, uint8_t* sc,
                               uint8_t* m, int N, int K, cudaStream_t st) {
    long long sbs = (long long)N * (K / 256);
    long long blocks = (sbs + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    quantize_k4_kernel<<<(unsigned)blocks, 256, 0, st>>>(w, codes, d, dmin, sc, m, N, K);
    return cudaGetLastError();
}

}  // namespace uq
