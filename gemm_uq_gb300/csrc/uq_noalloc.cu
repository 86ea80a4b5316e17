// uq_noalloc.cu -- uq_gemm_noalloc: the small-M GEMV with its scratch in a static device array.
//
// uq_gemm keeps its split-K scratch (fp32 partial sums and per-row-block tickets) in buffers the
// library allocates with cudaMalloc on first use.  Some callers cannot let a library allocate:
// a serving runtime that reserves the whole device memory up front and hands out nothing after
// start-up (cudaMalloc would fail there, or take memory the runtime already promised elsewhere),
// and latency-critical loops in which the implicit device synchronisation of cudaMalloc/cudaFree
// is not acceptable.  This entry point runs the same GEMV kernel with the scratch placed in a
// file-scope __device__ array of fixed size, so it calls no allocator at all.
#include <cstdio>
#include <mutex>

#include "uq_kernels.h"

namespace {

// Scratch layout (bytes): [0, 256) fault word; [256, 256 + TICKET_BYTES) row-block tickets;
// then the fp32 partial sums.  Every GPU that loads the library holds this array until exit.
constexpr size_t SCRATCH_BYTES = 1u << 20;                 // 1 MiB
constexpr size_t TICKET_BYTES = 256u << 10;                // 65536 row blocks of 16 = N <= 1048576
constexpr size_t PARTIAL_OFFSET = 256 + TICKET_BYTES;
constexpr size_t PARTIAL_BYTES = SCRATCH_BYTES - PARTIAL_OFFSET;

static __device__ __align__(256) unsigned char g_noalloc_scratch[SCRATCH_BYTES];

// Device address of the array, looked up once per device (host code cannot use the symbol's
// name as a device pointer: in host code it names a host-side shadow object).
std::mutex g_mu;
void* g_scratch_ptr[64] = {};
int g_sms[64] = {};

// message of the last failure on the calling thread, reported through uq_last_error()
thread_local char g_err[256] = "";
uq_status err(uq_status s) {
    uq::set_last_error(g_err);
    return s;
}

uq_status setup(int* dev_out, unsigned char** scratch, int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { snprintf(g_err, sizeof g_err, "cudaGetDevice: %s", cudaGetErrorString(e)); return err(UQ_ERR_CUDA); }
    if (dev < 0 || dev >= 64) { snprintf(g_err, sizeof g_err, "device index %d out of range", dev); return err(UQ_ERR_CUDA); }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        int major = 0, minor = 0, n = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3) {
            snprintf(g_err, sizeof g_err, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                     minor);
            return err(UQ_ERR_UNSUPPORTED);
        }
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) { snprintf(g_err, sizeof g_err, "SM count: %s", cudaGetErrorString(e)); return err(UQ_ERR_CUDA); }
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            snprintf(g_err, sizeof g_err, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
            return err(UQ_ERR_CUDA);
        }
        g_sms[dev] = n;
        g_scratch_ptr[dev] = p;
    }
    *dev_out = dev;
    *scratch = static_cast<unsigned char*>(g_scratch_ptr[dev]);
    *sms = g_sms[dev];
    return UQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

uq_status uq_gemm_noalloc(const uint16_t* x, const void* wq, const void* scales, const void* zeros_or_codebook,
                          uint16_t* y, int M, int N, int K, int group, uq_fmt fmt, void* stream) {
    g_err[0] = 0;
    if (fmt < UQ_INT4_SYM || fmt > UQ_K4) { snprintf(g_err, sizeof g_err, "unknown format"); return err(UQ_ERR_INVALID); }
    if (M < 0 || N < 0 || K < 0) { snprintf(g_err, sizeof g_err, "negative size"); return err(UQ_ERR_INVALID); }
    if (fmt == UQ_K4) {
        if (group != 256) { snprintf(g_err, sizeof g_err, "UQ_K4 needs group 256"); return err(UQ_ERR_UNSUPPORTED); }
        if (K % 256) { snprintf(g_err, sizeof g_err, "UQ_K4 needs K %% 256 == 0"); return err(UQ_ERR_INVALID); }
    } else {
        if (group != 32 && group != 64 && group != 128) {
            snprintf(g_err, sizeof g_err, "group must be 32, 64 or 128");
            return err(UQ_ERR_UNSUPPORTED);
        }
        if (K % group) { snprintf(g_err, sizeof g_err, "K is not a multiple of the group"); return err(UQ_ERR_INVALID); }
        if (fmt == UQ_INT2_ASYM && (K % 64)) {
            snprintf(g_err, sizeof g_err, "UQ_INT2_ASYM needs K %% 64 == 0");
            return err(UQ_ERR_UNSUPPORTED);
        }
    }
    if (M == 0 || N == 0 || K == 0) {
        // K == 0 would need a fill of y; keep this entry point to the kernel itself
        if (K == 0 && M > 0 && N > 0) { snprintf(g_err, sizeof g_err, "K == 0 is not supported here"); return err(UQ_ERR_UNSUPPORTED); }
        return UQ_OK;
    }
    const bool needs_zc = (fmt == UQ_INT4_ASYM || fmt == UQ_INT2_ASYM || fmt == UQ_NF4);
    if (!x || !wq || !scales || !y || (needs_zc != (zeros_or_codebook != nullptr))) {
        snprintf(g_err, sizeof g_err, "null pointer, or zeros_or_codebook given/missing for this format");
        return err(UQ_ERR_INVALID);
    }
    if (!aligned16(x) || !aligned16(wq) || !aligned16(scales) || !aligned16(y) ||
        (zeros_or_codebook && !aligned16(zeros_or_codebook))) {
        snprintf(g_err, sizeof g_err, "pointers must be 16-byte aligned");
        return err(UQ_ERR_ALIGN);
    }
    int dev = 0, sms = 0;
    unsigned char* scratch = nullptr;
    uq_status s = setup(&dev, &scratch, &sms);
    if (s != UQ_OK) return s;

    const uq::Layout L(N, K, fmt);
    const long long T = (long long)L.NB * L.KB;
    const int warps = uq::gemv_warps(fmt);
    long long P = (long long)sms * uq::gemv_ctas_per_sm(fmt) * warps;
    if (P > T) P = T;
    const int mb_max = M < 8 ? M : 8;
    if ((size_t)L.NB * sizeof(unsigned int) > TICKET_BYTES ||
        uq::gemv_partials_floats(fmt, T, (int)P, mb_max) * sizeof(float) > PARTIAL_BYTES) {
        snprintf(g_err, sizeof g_err,
                 "N=%d, M=%d needs more than the %zu-byte static scratch (at most %zu row blocks of 16 and "
                 "%zu bytes of partial sums)", N, M, SCRATCH_BYTES, TICKET_BYTES / 4, PARTIAL_BYTES);
        return err(UQ_ERR_NOMEM);
    }
    if (uq::gemv_smem_bytes(fmt, K, group, mb_max) > 227 * 1024) {
        snprintf(g_err, sizeof g_err, "K=%d is too long for the GEMV at M=%d", K, mb_max);
        return err(UQ_ERR_UNSUPPORTED);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int* tickets = reinterpret_cast<unsigned int*>(scratch + 256);
    float* partials = reinterpret_cast<float*>(scratch + PARTIAL_OFFSET);
    // the tickets must start at zero; the array keeps whatever the previous call left
    cudaError_t e = cudaMemsetAsync(tickets, 0, (size_t)L.NB * sizeof(unsigned int), st);
    if (e != cudaSuccess) { snprintf(g_err, sizeof g_err, "clearing tickets: %s", cudaGetErrorString(e)); return err(UQ_ERR_CUDA); }
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mb = (M - m0) < 8 ? (M - m0) : 8;
        uq::GemvArgs a;
        a.x = x + (long long)m0 * K;
        a.wq = static_cast<const uint8_t*>(wq);
        a.scales = static_cast<const uint8_t*>(scales);
        a.zc = static_cast<const uint8_t*>(zeros_or_codebook);
        a.y = y + (long long)m0 * N;
        a.M = mb; a.N = N; a.K = K; a.group = group; a.ldx = K; a.ldy = N;
        a.NB = L.NB; a.KB = L.KB; a.T = T; a.P = (int)P;
        a.partials = partials;
        a.tickets = tickets;
        a.fault = reinterpret_cast<unsigned int*>(scratch);
        a.overlap = 0;
        const int grid = uq::gemv_grid(a, fmt, sms);
        e = uq::launch_gemv(fmt, a, grid, st);
        if (e != cudaSuccess) { snprintf(g_err, sizeof g_err, "GEMV launch: %s", cudaGetErrorString(e)); return err(UQ_ERR_CUDA); }
    }
    return UQ_OK;
}

}  // extern "C"
