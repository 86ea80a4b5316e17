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

// Scratch layout (bytes): [0, 256) the fault word of no-alloc launches; from 256 the row-block
// tickets of the CUDA-core GEMV (INT8_SYM, NF4; 4 bytes per 16-row block, rounded up to 256 bytes),
// then the fp32 partial sums of row blocks split between workers.  A launch uses tickets and partial
// sums only when its work split needs them, so the limit depends on the shape (see uq.h).
// Every GPU that loads the library holds this array until the process exits.
constexpr size_t SCRATCH_BYTES = 1u << 20;                 // 1 MiB
constexpr size_t DATA_OFFSET = 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[SCRATCH_BYTES];

// Device address of the array, looked up once per device (host code cannot use the symbol's
// name as a device pointer: in host code it names a host-side shadow object).
std::mutex g_mu;
void* g_scratch_ptr[64] = {};
int g_sms[64] = {};

// message of the last failure on the calling thread, reported through uq_last_error()
thread_local char g_err[320] = "";
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
size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// the shape rules of uq_gemm_noalloc (those of uq_gemm's GEMV)
uq_status check_shape(int M, int N, int K, int group, uq_fmt fmt) {
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
    return UQ_OK;
}

// The scratch a call needs: the work split of its launches (every 8-row block of x but a shorter last
// one plans alike: the split depends on N and K, and the scratch it needs grows with the rows).
struct ScratchNeed {
    bool tickets;
    size_t ticket_bytes, partial_bytes;
};
uq_status scratch_need(int M, int N, int K, int group, uq_fmt fmt, int sms, ScratchNeed* need) {
    const uq::Layout L(N, K, fmt);
    const int mb_max = M < 8 ? M : 8;
    uq::GemvArgs probe = {};
    probe.M = mb_max; probe.N = N; probe.K = K; probe.group = group;
    probe.NB = L.NB; probe.KB = L.KB; probe.T = (long long)L.NB * L.KB;
    if (uq::gemv_plan(probe, fmt, sms) == 0) {
        snprintf(g_err, sizeof g_err, "K=%d is too long for the GEMV at M=%d", K, mb_max);
        return err(UQ_ERR_UNSUPPORTED);
    }
    need->tickets = uq::gemv_uses_tickets(fmt, probe);
    need->ticket_bytes = need->tickets ? round256((size_t)L.NB * sizeof(unsigned int)) : 0;
    need->partial_bytes = uq::gemv_partials_floats(fmt, probe) * sizeof(float);
    return UQ_OK;
}

}  // namespace

namespace uq {

// Reads and clears the fault word of no-alloc launches on the current device (the first word of the
// static array: the same address uq_gemm_noalloc hands its kernels).  *v = 0 when no no-alloc call
// ran on this device.  Synchronous; allocates nothing.
cudaError_t noalloc_take_fault(unsigned int* v) {
    *v = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    void* p = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        p = g_scratch_ptr[dev];
    }
    if (!p) return cudaSuccess;
    e = cudaMemcpy(v, p, sizeof(unsigned int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess || *v == 0) return e;
    // a launch gave up early: clear the word (every call clears the tickets it uses itself)
    return cudaMemset(p, 0, sizeof(unsigned int));
}

}  // namespace uq

extern "C" {

uq_status uq_gemm_noalloc(const uint16_t* x, const void* wq, const void* scales, const void* zeros_or_codebook,
                          uint16_t* y, int M, int N, int K, int group, uq_fmt fmt, void* stream) {
    g_err[0] = 0;
    uq_status s0 = check_shape(M, N, K, group, fmt);
    if (s0 != UQ_OK) return s0;
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
    ScratchNeed need;
    if ((s = scratch_need(M, N, K, group, fmt, sms, &need)) != UQ_OK) return s;
    const bool uses_tickets = need.tickets;
    const size_t ticket_bytes = need.ticket_bytes, partial_bytes = need.partial_bytes;
    if (DATA_OFFSET + ticket_bytes + partial_bytes > SCRATCH_BYTES) {
        snprintf(g_err, sizeof g_err,
                 "M=%d, N=%d, K=%d needs %zu bytes of tickets and %zu bytes of partial sums; the static scratch "
                 "holds %zu bytes in all", M, N, K, ticket_bytes, partial_bytes, SCRATCH_BYTES - DATA_OFFSET);
        return err(UQ_ERR_NOMEM);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int* tickets = reinterpret_cast<unsigned int*>(scratch + DATA_OFFSET);
    float* partials = reinterpret_cast<float*>(scratch + DATA_OFFSET + ticket_bytes);
    cudaError_t e = cudaSuccess;
    if (uses_tickets) {
        // the tickets must start at zero; the array keeps whatever the previous call left
        e = cudaMemsetAsync(tickets, 0, (size_t)L.NB * sizeof(unsigned int), st);
        if (e != cudaSuccess) { snprintf(g_err, sizeof g_err, "clearing tickets: %s", cudaGetErrorString(e)); return err(UQ_ERR_CUDA); }
    }
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mb = (M - m0) < 8 ? (M - m0) : 8;
        uq::GemvArgs a = {};
        a.x = x + (long long)m0 * K;
        a.wq = static_cast<const uint8_t*>(wq);
        a.scales = static_cast<const uint8_t*>(scales);
        a.zc = static_cast<const uint8_t*>(zeros_or_codebook);
        a.y = y + (long long)m0 * N;
        a.M = mb; a.N = N; a.K = K; a.group = group; a.ldx = K; a.ldy = N;
        a.NB = L.NB; a.KB = L.KB; a.T = T;
        const int grid = uq::gemv_plan(a, fmt, sms);
        a.partials = partials;
        a.tickets = tickets;
        a.fault = reinterpret_cast<unsigned int*>(scratch);     // read back by uq_device_fault
        a.overlap = 0;
        e = uq::launch_gemv(fmt, a, grid, st);
        if (e != cudaSuccess) { snprintf(g_err, sizeof g_err, "GEMV launch: %s", cudaGetErrorString(e)); return err(UQ_ERR_CUDA); }
    }
    return UQ_OK;
}

uq_status uq_gemm_noalloc_scratch(int M, int N, int K, int group, uq_fmt fmt, size_t* ticket_bytes,
                                  size_t* partial_bytes) {
    g_err[0] = 0;
    if (!ticket_bytes || !partial_bytes) { snprintf(g_err, sizeof g_err, "null pointer"); return err(UQ_ERR_INVALID); }
    *ticket_bytes = *partial_bytes = 0;
    uq_status s = check_shape(M, N, K, group, fmt);
    if (s != UQ_OK) return s;
    if (M == 0 || N == 0 || K == 0) return UQ_OK;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms < 1) {
        snprintf(g_err, sizeof g_err, "SM count: %s", cudaGetErrorString(e != cudaSuccess ? e : cudaErrorInvalidDevice));
        return err(UQ_ERR_CUDA);
    }
    ScratchNeed need;
    if ((s = scratch_need(M, N, K, group, fmt, sms, &need)) != UQ_OK) return s;
    *ticket_bytes = need.ticket_bytes;
    *partial_bytes = need.partial_bytes;
    return UQ_OK;
}

}  // extern "C"
