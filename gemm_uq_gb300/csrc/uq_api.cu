// uq_api.cu -- the C ABI (include/uq.h): argument validation, path choice, workspace, launches.
//
// Host-side only.  Every entry point validates its arguments and returns a status; nothing
// throws across the ABI and nothing falls back to another implementation: a request the
// kernels do not implement is refused with UQ_ERR_UNSUPPORTED.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "uq_kernels.h"

namespace {

constexpr int RB_ROWS = 16;   // rows per row block of the packed plane
thread_local std::string g_last_error = "";

uq_status fail(uq_status s, const char* fmt_msg, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt_msg);
    vsnprintf(buf, sizeof buf, fmt_msg, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

uq_status cuda_fail(cudaError_t e, const char* what) {
    return fail(UQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_fmt(int fmt) { return fmt >= UQ_INT4_SYM && fmt <= UQ_K4; }

// shape rules shared by every call that takes (N, K, group, fmt)
uq_status check_shape(int N, int K, int group, int fmt) {
    if (!valid_fmt(fmt)) return fail(UQ_ERR_INVALID, "unknown format %d", fmt);
    if (N < 0 || K < 0) return fail(UQ_ERR_INVALID, "negative size N=%d K=%d", N, K);
    if (fmt == UQ_K4) {
        if (group != 256) return fail(UQ_ERR_UNSUPPORTED, "UQ_K4 needs group 256 (got %d)", group);
        if (K % 256) return fail(UQ_ERR_INVALID, "UQ_K4 needs K %% 256 == 0 (K=%d)", K);
        return UQ_OK;
    }
    if (group != 32 && group != 64 && group != 128)
        return fail(UQ_ERR_UNSUPPORTED, "group must be 32, 64 or 128 (got %d)", group);
    if (K % group) return fail(UQ_ERR_INVALID, "K=%d is not a multiple of group %d", K, group);
    if (fmt == UQ_INT2_ASYM && (K % 64))
        return fail(UQ_ERR_UNSUPPORTED, "UQ_INT2_ASYM needs K %% 64 == 0 (K=%d)", K);
    return UQ_OK;
}

size_t meta_scales_bytes(int N, int K, int group, int fmt) {
    if (fmt == UQ_K4) return (size_t)N * (K / 256) * 16;
    return (size_t)N * (K / group) * 2;
}
size_t meta_zeros_bytes(int N, int K, int group, int fmt) {
    if (fmt == UQ_INT4_ASYM) return (size_t)N * ((K / group + 1) / 2);
    if (fmt == UQ_INT2_ASYM) return (size_t)N * (K / group) * 2;
    if (fmt == UQ_NF4) return 64;
    return 0;
}
bool needs_zc(int fmt) { return fmt == UQ_INT4_ASYM || fmt == UQ_INT2_ASYM || fmt == UQ_NF4; }

// ---------------------------------------------------------------------------------------------
// per-device state: SM count and two device words (fault flag, pack range violations)
struct DeviceState {
    int sms = 0;
    unsigned int* words = nullptr;   // [0] fault, [1] bad-code counter
};
std::mutex g_mu;
std::map<int, DeviceState> g_dev;

// per (device, stream) workspace for the split-K partial sums and the row-block tickets
struct Workspace {
    float* partials = nullptr;
    size_t partial_bytes = 0;
    float* aux = nullptr;              // K4 GEMMs: column sums of x per 32-k block; W4A8: x codes
    size_t aux_bytes = 0;
    unsigned int* tickets = nullptr;   // zero between calls (the kernels reset what they use)
    size_t ticket_bytes = 0;
    float* gate32 = nullptr;           // gated projection: fp32 gate outputs [M][N]
    size_t gate32_bytes = 0;
};
std::map<std::pair<int, void*>, Workspace> g_ws;

// Workspace buffers replaced by a larger one.  They are never freed: a CUDA graph captured before
// the growth still holds their addresses and may be replayed at any time, so they stay allocated
// (and their tickets zero) until the process exits.  Growth doubles, so they add up to less than
// the buffer that replaced them.
struct Retired {
    int dev;
    void* ptr;
    size_t bytes;
    bool tickets;
};
std::vector<Retired> g_retired;

uq_status device_state(DeviceState** out, int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.words) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(UQ_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                        major, minor);
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        e = cudaMalloc(&d.words, 256);
        if (e != cudaSuccess) return fail(UQ_ERR_NOMEM, "cudaMalloc of device words failed");
        e = cudaMemset(d.words, 0, 256);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
    }
    *out = &d;
    if (dev_out) *dev_out = dev;
    return UQ_OK;
}

uq_status grow(void** ptr, size_t* have, size_t need, bool zero, cudaStream_t st, int dev) {
    if (*have >= need) return UQ_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
        return fail(UQ_ERR_NOMEM, "workspace must grow to %zu bytes but the stream is being captured; "
                                  "make one call of this size before capturing", need);
    size_t bytes = *have ? *have : 4096;
    while (bytes < need) bytes *= 2;
    void* fresh = nullptr;
    e = cudaMalloc(&fresh, bytes);
    if (e != cudaSuccess) return fail(UQ_ERR_NOMEM, "cudaMalloc(%zu) failed", bytes);
    if (*ptr) g_retired.push_back({dev, *ptr, *have, zero});   // graphs captured earlier may still use it
    *ptr = fresh;
    if (zero) {
        e = cudaMemsetAsync(*ptr, 0, bytes, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    }
    *have = bytes;
    return UQ_OK;
}

uq_status workspace(int dev, cudaStream_t st, size_t partial_bytes, size_t ticket_bytes, Workspace** out,
                    size_t aux_bytes = 0) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace& w = g_ws[{dev, (void*)st}];
    uq_status s = grow(reinterpret_cast<void**>(&w.partials), &w.partial_bytes, partial_bytes, false, st, dev);
    if (s != UQ_OK) return s;
    if (aux_bytes) {
        s = grow(reinterpret_cast<void**>(&w.aux), &w.aux_bytes, aux_bytes, false, st, dev);
        if (s != UQ_OK) return s;
    }
    s = grow(reinterpret_cast<void**>(&w.tickets), &w.ticket_bytes, ticket_bytes, true, st, dev);
    if (s != UQ_OK) return s;
    *out = &w;
    return UQ_OK;
}

// Output mode of a launch: plain bf16 y; or the gated projection's gate pass (fp32 into out32) or up
// pass (bf16 silu(gate32) * result into y)
struct OutMode {
    float* out32 = nullptr;
    const float* gate32 = nullptr;
};

// one GEMV launch for Mb <= 8 rows of x
uq_status run_gemv(const uint16_t* x, const void* wq, const void* scales, const void* zc, uint16_t* y,
                   int Mb, int N, int K, int ldx, int ldy, int group, int fmt, cudaStream_t st,
                   const DeviceState& ds, int dev, OutMode om = OutMode()) {
    const uq::Layout L(N, K, fmt);
    uq::GemvArgs a = {};
    a.M = Mb; a.N = N; a.K = K; a.group = group; a.ldx = ldx; a.ldy = ldy;
    a.NB = L.NB; a.KB = L.KB; a.T = (long long)L.NB * L.KB;
    const int grid = uq::gemv_plan(a, fmt, ds.sms);
    if (grid == 0)
        return fail(UQ_ERR_UNSUPPORTED, "K=%d is too long for the GEMV's shared memory at M=%d", K, Mb);
    Workspace* ws = nullptr;
    uq_status s = workspace(dev, st, uq::gemv_partials_floats(fmt, a) * sizeof(float),
                            (size_t)L.NB * sizeof(unsigned int), &ws);
    if (s != UQ_OK) return s;
    a.x = x;
    a.wq = static_cast<const uint8_t*>(wq);
    a.scales = static_cast<const uint8_t*>(scales);
    a.zc = static_cast<const uint8_t*>(zc);
    a.y = y;
    a.partials = ws->partials;
    a.tickets = ws->tickets;
    a.fault = ds.words;
    a.out32 = om.out32;
    a.gate32 = om.gate32;
    cudaError_t e = uq::launch_gemv(fmt, a, grid, st);
    if (e != cudaSuccess) return cuda_fail(e, "GEMV launch");
    return UQ_OK;
}


// the gated projection for Mb <= 8 rows of x in one mma-GEMV launch: gate and up row blocks
// interleaved in one work list, every CTA owning whole gate/up pairs
uq_status run_gemv_gated(const uint16_t* x, const void* wg, const void* sg, const void* zg, const void* wu,
                         const void* su, const void* zu, uint16_t* h, int Mb, int N, int K, int ldx, int ldy,
                         int group, int fmt, cudaStream_t st, const DeviceState& ds, int dev) {
    const uq::Layout L(N, K, fmt);
    uq::GemvArgs a = {};
    a.gated = 1;
    a.M = Mb; a.N = N; a.K = K; a.group = group; a.ldx = ldx; a.ldy = ldy;
    a.NB = 2 * L.NB; a.KB = L.KB; a.T = 2LL * L.NB * L.KB;
    const int grid = uq::gemv_plan(a, fmt, ds.sms);
    if (grid == 0)
        return fail(UQ_ERR_UNSUPPORTED, "K=%d is too long for the GEMV's shared memory at M=%d", K, Mb);
    Workspace* ws = nullptr;
    uq_status s = workspace(dev, st, uq::gemv_partials_floats(fmt, a) * sizeof(float),
                            (size_t)L.NB * sizeof(unsigned int), &ws);
    if (s != UQ_OK) return s;
    a.x = x;
    a.wq = static_cast<const uint8_t*>(wg);
    a.scales = static_cast<const uint8_t*>(sg);
    a.zc = static_cast<const uint8_t*>(zg);
    a.wq2 = static_cast<const uint8_t*>(wu);
    a.scales2 = static_cast<const uint8_t*>(su);
    a.zc2 = static_cast<const uint8_t*>(zu);
    a.y = h;
    a.partials = ws->partials;
    a.tickets = ws->tickets;
    a.fault = ds.words;
    cudaError_t e = uq::launch_gemv(fmt, a, grid, st);
    if (e != cudaSuccess) return cuda_fail(e, "gated GEMV launch");
    return UQ_OK;
}

// one tensor-core launch for 16 <= Mb <= 64 rows of x
uq_status run_tc(const uint16_t* x, const void* wq, const void* scales, const void* zc, uint16_t* y, int Mb, int N,
                 int K, int ldx, int ldy, int group, int fmt, cudaStream_t st, const DeviceState& ds, int dev,
                 OutMode om = OutMode()) {
    const int mpad = (Mb + 15) / 16 * 16;
    size_t smem = 0;
    if (uq::tc_plan(fmt, mpad, group, &smem) != 0)
        return fail(UQ_ERR_UNSUPPORTED, "no tensor-core plan for M=%d", Mb);
    const int kc = (fmt == UQ_INT8_SYM || fmt == UQ_NF4) ? 128 : 256;   // codes per row per unit
    const int nblk = (N + 127) / 128;
    const int CH = K / kc;
    const long long U = (long long)nblk * CH;
    long long P = ds.sms;
    if (P > U) P = U;
    Workspace* ws = nullptr;
    const size_t aux = (fmt == UQ_K4) ? (size_t)(K / 32) * mpad * sizeof(float) : 0;
    uq_status s = workspace(dev, st, (size_t)2 * P * 128 * mpad * sizeof(float), (size_t)nblk * sizeof(unsigned int),
                            &ws, aux);
    if (s != UQ_OK) return s;
    cudaError_t e;
    if (fmt == UQ_K4) {
        e = uq::launch_colsum32(x, ws->aux, Mb, mpad, K, ldx, st);
        if (e != cudaSuccess) return cuda_fail(e, "column-sum launch");
    }
    uq::TcArgs a = {};
    const uq::Layout L(N, K, fmt);
    a.wq = static_cast<const uint8_t*>(wq);
    a.rowbytes = L.rowbytes;
    a.NB = L.NB;
    a.scales = static_cast<const uint8_t*>(scales);
    a.zc = static_cast<const uint8_t*>(zc);
    a.y = y;
    a.sx = ws->aux;
    a.M = Mb; a.Mpad = mpad; a.N = N; a.K = K; a.group = group; a.ldx = ldx; a.ldy = ldy;
    a.CH = CH; a.U = U; a.P = (int)P;
    a.partials = ws->partials;
    a.tickets = ws->tickets;
    a.fault = ds.words;
    a.out32 = om.out32;
    a.gate32 = om.gate32;
    e = uq::launch_tc(fmt, x, a, smem, (int)P, st);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-core launch");
    return UQ_OK;
}


// one mma.sync GEMM launch (and its second pass when the k range is split) for 9 <= Mb <= 64 rows
// of x, 4-bit and 2-bit formats
uq_status run_gemm_mma(const uint16_t* x, const void* wq, const void* scales, const void* zc, uint16_t* y, int Mb,
                       int N, int K, int ldx, int ldy, int group, int fmt, cudaStream_t st, const DeviceState& ds,
                       int dev, OutMode om = OutMode()) {
    const uq::Layout L(N, K, fmt);
    uq::GemmArgs a = {};
    a.M = Mb; a.N = N; a.K = K; a.group = group; a.ldx = ldx; a.ldy = ldy;
    a.NB = L.NB;
    a.UB = uq::gemm_mma_units(fmt, K);
    a.KS = uq::gemm_mma_splits(a.NB, a.UB, ds.sms);
    a.Mpad = Mb <= 16 ? 16 : (Mb <= 32 ? 32 : 64);
    const size_t partial_bytes = a.KS > 1 ? (size_t)a.KS * a.NB * 16 * Mb * sizeof(float) : 0;
    const size_t aux_bytes = (fmt == UQ_K4) ? (size_t)(K / 32) * a.Mpad * sizeof(float) : 0;
    Workspace* ws = nullptr;
    uq_status s = workspace(dev, st, partial_bytes, (size_t)L.NB * sizeof(unsigned int), &ws, aux_bytes);
    if (s != UQ_OK) return s;
    cudaError_t e;
    if (fmt == UQ_K4) {
        e = uq::launch_colsum32(x, ws->aux, Mb, a.Mpad, K, ldx, st);
        if (e != cudaSuccess) return cuda_fail(e, "column-sum launch");
    }
    a.x = x;
    a.wq = static_cast<const uint8_t*>(wq);
    a.scales = static_cast<const uint8_t*>(scales);
    a.zc = static_cast<const uint8_t*>(zc);
    a.y = y;
    a.sx = ws->aux;
    a.partials = ws->partials;
    a.out32 = om.out32;
    a.gate32 = om.gate32;
    e = uq::launch_gemm_mma(fmt, a, ds.sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "mma GEMM launch");
    return UQ_OK;
}

// Which kernel runs a block of rows of x (automatic choice, from measurements of both GEMMs): the
// 4-bit and 2-bit formats take the mma.sync GEMM for 9..15 rows (instead of two 8-row GEMV passes
// over the weights) and K4 for any M >= 9; every format takes the tensor-core GEMM for 16..64 rows
// otherwise, when the shape allows it; everything else runs the GEMV in blocks of at most 8 rows.
// uq_set_gemm_path can force either GEMM for M >= 16.
std::atomic<int> g_path{0};                 // uq_set_gemm_path: 0 automatic, 1 tensor cores, 2 mma.sync
enum Route { ROUTE_GEMV = 0, ROUTE_MMA_GEMM = 1, ROUTE_TC = 2 };
Route route(int fmt, int M, int N, int K) {
    const int path = g_path.load(std::memory_order_relaxed);
    const bool tc = M >= 16 && uq::tc_supported(fmt, N, K);
    if (uq::gemm_mma_format(fmt) && M >= 9) {
        if (path == 2) return ROUTE_MMA_GEMM;
        if (path == 1 && tc) return ROUTE_TC;
        if (path == 0 && (M <= 15 || fmt == UQ_K4 || !tc)) return ROUTE_MMA_GEMM;
    }
    return tc ? ROUTE_TC : ROUTE_GEMV;
}
// launches of one mma.sync GEMM block of Mb rows
int gemm_mma_launches(int fmt, int Mb, int N, int K, int sms) {
    const uq::Layout L(N, K, fmt);
    const int ks = uq::gemm_mma_splits(L.NB, uq::gemm_mma_units(fmt, K), sms);
    (void)Mb;
    return 1 + (ks > 1 ? 1 : 0) + (fmt == UQ_K4 ? 1 : 0);
}
}  // namespace

namespace uq {
void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }
static std::atomic<int> g_overlap{0};
bool launch_overlap() { return g_overlap.load(std::memory_order_relaxed) != 0; }
}  // namespace uq

// =============================================================================================
extern "C" {

const char* uq_status_string(uq_status s) {
    switch (s) {
        case UQ_OK: return "UQ_OK";
        case UQ_ERR_INVALID: return "UQ_ERR_INVALID";
        case UQ_ERR_UNSUPPORTED: return "UQ_ERR_UNSUPPORTED";
        case UQ_ERR_ALIGN: return "UQ_ERR_ALIGN";
        case UQ_ERR_CUDA: return "UQ_ERR_CUDA";
        case UQ_ERR_NOMEM: return "UQ_ERR_NOMEM";
        default: return "UQ_ERR_UNKNOWN";
    }
}

const char* uq_last_error(void) { return g_last_error.c_str(); }

uq_status uq_packed_size(int N, int K, int group, uq_fmt fmt, size_t* wq_bytes, size_t* scales_bytes,
                         size_t* zeros_bytes) {
    uq_status s = check_shape(N, K, group, fmt);
    if (s != UQ_OK) return s;
    if (wq_bytes) *wq_bytes = (size_t)uq::Layout(N, K, fmt).bytes();
    if (scales_bytes) *scales_bytes = meta_scales_bytes(N, K, group, fmt);
    if (zeros_bytes) *zeros_bytes = meta_zeros_bytes(N, K, group, fmt);
    return UQ_OK;
}

uq_status uq_pack_layout(const int8_t* codes, void* wq, int N, int K, int group, uq_fmt fmt, void* stream) {
    uq_status s = check_shape(N, K, group, fmt);
    if (s != UQ_OK) return s;
    if ((long long)N * K == 0) return UQ_OK;
    if (!codes || !wq) return fail(UQ_ERR_INVALID, "null pointer");
    if (!aligned16(codes) || !aligned16(wq)) return fail(UQ_ERR_ALIGN, "codes and wq must be 16-byte aligned");
    DeviceState* ds = nullptr;
    if ((s = device_state(&ds, nullptr)) != UQ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(ds->words + 1, 0, sizeof(unsigned int), st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    e = uq::launch_pack(fmt, codes, static_cast<uint8_t*>(wq), N, K, ds->words + 1, st);
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    unsigned int bad = 0;
    e = cudaMemcpyAsync(&bad, ds->words + 1, sizeof bad, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "pack check");
    if (bad) return fail(UQ_ERR_INVALID, "%u code words hold a code outside the format's range", bad);
    return UQ_OK;
}

uq_status uq_pack_kmeta(const uint16_t* d, const uint16_t* dmin, const uint8_t* sc, const uint8_t* m, void* meta,
                        int N, int K, void* stream) {
    uq_status s = check_shape(N, K, 256, UQ_K4);
    if (s != UQ_OK) return s;
    const long long count = (long long)N * (K / 256);
    if (count == 0) return UQ_OK;
    if (!d || !dmin || !sc || !m || !meta) return fail(UQ_ERR_INVALID, "null pointer");
    if (!aligned16(d) || !aligned16(dmin) || !aligned16(sc) || !aligned16(m) || !aligned16(meta))
        return fail(UQ_ERR_ALIGN, "K4 metadata pointers must be 16-byte aligned");
    DeviceState* ds = nullptr;
    if ((s = device_state(&ds, nullptr)) != UQ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(ds->words + 1, 0, sizeof(unsigned int), st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    e = uq::launch_pack_kmeta(d, dmin, sc, m, static_cast<uint8_t*>(meta), count, ds->words + 1, st);
    if (e != cudaSuccess) return cuda_fail(e, "kmeta launch");
    unsigned int bad = 0;
    e = cudaMemcpyAsync(&bad, ds->words + 1, sizeof bad, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "kmeta check");
    if (bad) return fail(UQ_ERR_INVALID, "%u K4 records hold a 6-bit code above 63", bad);
    return UQ_OK;
}

uq_status uq_pack_zeros(const uint8_t* zeros, uint8_t* packed, int N, int G, void* stream) {
    if (N < 0 || G < 0) return fail(UQ_ERR_INVALID, "negative size");
    if ((long long)N * G == 0) return UQ_OK;
    if (!zeros || !packed) return fail(UQ_ERR_INVALID, "null pointer");
    if (!aligned16(zeros) || !aligned16(packed)) return fail(UQ_ERR_ALIGN, "pointers must be 16-byte aligned");
    cudaError_t e = uq::launch_pack_zeros(zeros, packed, N, G, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pack_zeros launch");
    return UQ_OK;
}

static uq_status check_meta_ptrs(const void* scales, const void* zc, int fmt) {
    if (!scales) return fail(UQ_ERR_INVALID, "scales is NULL");
    if (needs_zc(fmt) && !zc) return fail(UQ_ERR_INVALID, "this format needs zeros_or_codebook");
    if (!needs_zc(fmt) && zc) return fail(UQ_ERR_INVALID, "zeros_or_codebook must be NULL for this format");
    if (!aligned16(scales) || (zc && !aligned16(zc)))
        return fail(UQ_ERR_ALIGN, "scales / zeros_or_codebook must be 16-byte aligned");
    return UQ_OK;
}

uq_status uq_gemm(const uint16_t* x, const void* wq, const void* scales, const void* zeros_or_codebook,
                  uint16_t* y, int M, int N, int K, int group, uq_fmt fmt, void* stream) {
    uq_status s = check_shape(N, K, group, fmt);
    if (s != UQ_OK) return s;
    if (M < 0) return fail(UQ_ERR_INVALID, "negative M");
    if (M == 0 || N == 0) return UQ_OK;
    if (!y) return fail(UQ_ERR_INVALID, "y is NULL");
    if (!aligned16(y)) return fail(UQ_ERR_ALIGN, "y must be 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, (size_t)M * N * 2, st);
        return e == cudaSuccess ? UQ_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (!x || !wq) return fail(UQ_ERR_INVALID, "x or wq is NULL");
    if (!aligned16(x) || !aligned16(wq)) return fail(UQ_ERR_ALIGN, "x and wq must be 16-byte aligned");
    if ((s = check_meta_ptrs(scales, zeros_or_codebook, fmt)) != UQ_OK) return s;
    DeviceState* ds = nullptr;
    int dev = 0;
    if ((s = device_state(&ds, &dev)) != UQ_OK) return s;
    const Route rt = route(fmt, M, N, K);
    if (rt == ROUTE_MMA_GEMM) {
        // blocks of at most 64 rows on the mma.sync GEMM; a last block of at most 8 rows on the GEMV
        for (int m0 = 0; m0 < M; m0 += 64) {
            const int mb = (M - m0) < 64 ? (M - m0) : 64;
            const uint16_t* xb = x + (long long)m0 * K;
            uint16_t* yb = y + (long long)m0 * N;
            s = mb <= 8 ? run_gemv(xb, wq, scales, zeros_or_codebook, yb, mb, N, K, K, N, group, fmt, st, *ds, dev)
                        : run_gemm_mma(xb, wq, scales, zeros_or_codebook, yb, mb, N, K, K, N, group, fmt, st, *ds, dev);
            if (s != UQ_OK) return s;
        }
        return UQ_OK;
    }
    if (rt == ROUTE_TC) {
        // tensor cores, in blocks of at most 64 activation rows (the last block at least 16 rows
        // wide is padded to a multiple of 16 with zero rows by the TMA bounds)
        for (int m0 = 0; m0 < M; m0 += 64) {
            const int mb = (M - m0) < 64 ? (M - m0) : 64;
            s = run_tc(x + (long long)m0 * K, wq, scales, zeros_or_codebook, y + (long long)m0 * N, mb, N, K, K, N,
                       group, fmt, st, *ds, dev);
            if (s != UQ_OK) return s;
        }
        return UQ_OK;
    }
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mb = (M - m0) < 8 ? (M - m0) : 8;
        s = run_gemv(x + (long long)m0 * K, wq, scales, zeros_or_codebook, y + (long long)m0 * N, mb, N, K, K, N,
                     group, fmt, st, *ds, dev);
        if (s != UQ_OK) return s;
    }
    return UQ_OK;
}

uq_status uq_gemm_gated(const uint16_t* x, const void* wq_gate, const void* scales_gate, const void* zc_gate,
                        const void* wq_up, const void* scales_up, const void* zc_up, uint16_t* h,
                        int M, int N, int K, int group, uq_fmt fmt, void* stream) {
    uq_status s = check_shape(N, K, group, fmt);
    if (s != UQ_OK) return s;
    if (M < 0) return fail(UQ_ERR_INVALID, "negative M");
    if (M == 0 || N == 0) return UQ_OK;
    if (!h) return fail(UQ_ERR_INVALID, "h is NULL");
    if (!aligned16(h)) return fail(UQ_ERR_ALIGN, "h must be 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K == 0) {   // g = u = 0, silu(0) * 0 = 0
        cudaError_t e = cudaMemsetAsync(h, 0, (size_t)M * N * 2, st);
        return e == cudaSuccess ? UQ_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (!x || !wq_gate || !wq_up) return fail(UQ_ERR_INVALID, "x, wq_gate or wq_up is NULL");
    if (!aligned16(x) || !aligned16(wq_gate) || !aligned16(wq_up))
        return fail(UQ_ERR_ALIGN, "x, wq_gate and wq_up must be 16-byte aligned");
    if ((s = check_meta_ptrs(scales_gate, zc_gate, fmt)) != UQ_OK) return s;
    if ((s = check_meta_ptrs(scales_up, zc_up, fmt)) != UQ_OK) return s;
    DeviceState* ds = nullptr;
    int dev = 0;
    if ((s = device_state(&ds, &dev)) != UQ_OK) return s;
    const Route rt = route(fmt, M, N, K);
    const bool tc = rt == ROUTE_TC;
    const int block = rt == ROUTE_GEMV ? 8 : 64;
    if (rt != ROUTE_TC && uq::gemv_is_mma(fmt) && M <= 8) {
        // one launch: the mma GEMV over the gate and up weights together
        return run_gemv_gated(x, wq_gate, scales_gate, zc_gate, wq_up, scales_up, zc_up, h, M, N, K, K, N, group,
                              fmt, st, *ds, dev);
    }
    const int rows = M < block ? M : block;
    float* g32 = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        Workspace& w = g_ws[{dev, (void*)st}];
        s = grow(reinterpret_cast<void**>(&w.gate32), &w.gate32_bytes, (size_t)rows * N * sizeof(float), false, st, dev);
        if (s != UQ_OK) return s;
        g32 = w.gate32;
    }
    // per block of rows of x: the gate projection into fp32 scratch, then the up projection, whose
    // epilogue writes h = bf16(silu(g) * u)
    for (int m0 = 0; m0 < M; m0 += block) {
        const int mb = (M - m0) < block ? (M - m0) : block;
        const uint16_t* xb = x + (long long)m0 * K;
        uint16_t* hb = h + (long long)m0 * N;
        OutMode gate_pass, up_pass;
        gate_pass.out32 = g32;
        up_pass.gate32 = g32;
        if (tc) {
            s = run_tc(xb, wq_gate, scales_gate, zc_gate, hb, mb, N, K, K, N, group, fmt, st, *ds, dev, gate_pass);
            if (s == UQ_OK)
                s = run_tc(xb, wq_up, scales_up, zc_up, hb, mb, N, K, K, N, group, fmt, st, *ds, dev, up_pass);
        } else if (rt == ROUTE_MMA_GEMM && mb <= 8) {
            s = run_gemv_gated(xb, wq_gate, scales_gate, zc_gate, wq_up, scales_up, zc_up, hb, mb, N, K, K, N, group,
                               fmt, st, *ds, dev);
        } else if (rt == ROUTE_MMA_GEMM) {
            s = run_gemm_mma(xb, wq_gate, scales_gate, zc_gate, hb, mb, N, K, K, N, group, fmt, st, *ds, dev, gate_pass);
            if (s == UQ_OK)
                s = run_gemm_mma(xb, wq_up, scales_up, zc_up, hb, mb, N, K, K, N, group, fmt, st, *ds, dev, up_pass);
        } else {
            s = run_gemv(xb, wq_gate, scales_gate, zc_gate, hb, mb, N, K, K, N, group, fmt, st, *ds, dev, gate_pass);
            if (s == UQ_OK)
                s = run_gemv(xb, wq_up, scales_up, zc_up, hb, mb, N, K, K, N, group, fmt, st, *ds, dev, up_pass);
        }
        if (s != UQ_OK) return s;
    }
    return UQ_OK;
}

uq_status uq_gemm_gated_kernel_count(int M, int N, int K, int group, uq_fmt fmt, int* count) {
    uq_status s = uq_gemm_kernel_count(M, N, K, group, fmt, count);
    if (s != UQ_OK || M == 0 || N == 0 || K == 0) return s;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms < 1) return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidDevice, "SM count");
    const Route rt = route(fmt, M, N, K);
    const uq::Layout L(N, K, fmt);
    // one fused GEMV launch for a block of at most 8 rows of a 4-bit / 2-bit format
    auto fused = [&](int mb) {
        uq::GemvArgs a = {};
        a.M = mb; a.N = N; a.K = K; a.group = group;
        a.gated = 1; a.NB = 2 * L.NB; a.KB = L.KB; a.T = (long long)a.NB * L.KB;
        uq::gemv_plan(a, fmt, sms);
        return uq::gemv_launches(fmt, a);
    };
    if (rt != ROUTE_TC && uq::gemv_is_mma(fmt) && M <= 8) {
        *count = fused(M);
        return UQ_OK;
    }
    if (rt == ROUTE_MMA_GEMM) {
        int n = 0;
        for (int m0 = 0; m0 < M; m0 += 64) {
            const int mb = (M - m0) < 64 ? (M - m0) : 64;
            n += mb <= 8 ? fused(mb) : 2 * gemm_mma_launches(fmt, mb, N, K, sms);   // a gate pass and an up pass
        }
        *count = n;
        return UQ_OK;
    }
    *count *= 2;                                            // the gate pass and the up pass
    return UQ_OK;
}

uq_status uq_rope_table(float* table, int max_pos, int head_dim, double base, void* stream) {
    if (max_pos < 0) return fail(UQ_ERR_INVALID, "negative max_pos");
    if (head_dim < 2 || head_dim % 2) return fail(UQ_ERR_INVALID, "head_dim must be even and positive (got %d)", head_dim);
    if (!(base > 1.0)) return fail(UQ_ERR_INVALID, "base must be above 1");
    if (max_pos == 0) return UQ_OK;
    if (!table) return fail(UQ_ERR_INVALID, "table is NULL");
    if (!aligned16(table)) return fail(UQ_ERR_ALIGN, "table must be 16-byte aligned");
    cudaError_t e = uq::launch_rope_table(table, max_pos, head_dim, base, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? UQ_OK : cuda_fail(e, "rope table launch");
}

uq_status uq_rmsnorm_rope(const uint16_t* x, const uint16_t* gamma, const int32_t* pos, const float* table,
                          uint16_t* y, int M, int D, int head_dim, int max_pos, float eps, void* stream) {
    if (M < 0 || D < 0 || max_pos < 0) return fail(UQ_ERR_INVALID, "negative size");
    if (head_dim < 16 || head_dim % 16)
        return fail(UQ_ERR_UNSUPPORTED, "head_dim must be a positive multiple of 16 (got %d)", head_dim);
    if (D % head_dim) return fail(UQ_ERR_INVALID, "D=%d is not a multiple of head_dim %d", D, head_dim);
    if (!(eps >= 0.0f)) return fail(UQ_ERR_INVALID, "eps must be >= 0");
    if (M == 0 || D == 0) return UQ_OK;
    if (!x || !gamma || !pos || !table || !y) return fail(UQ_ERR_INVALID, "null pointer");
    if (max_pos < 1) return fail(UQ_ERR_INVALID, "the rope table is empty");
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(table) || !aligned16(y) ||
        (reinterpret_cast<uintptr_t>(pos) & 3u))
        return fail(UQ_ERR_ALIGN, "x, gamma, table and y must be 16-byte aligned, pos 4-byte aligned");
    DeviceState* ds = nullptr;
    uq_status s = device_state(&ds, nullptr);
    if (s != UQ_OK) return s;
    cudaError_t e = uq::launch_rmsnorm_rope(x, gamma, pos, table, y, M, D, head_dim, max_pos, eps, ds->words, ds->sms,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? UQ_OK : cuda_fail(e, "rmsnorm_rope launch");
}

uq_status uq_pack_gguf(const void* blocks, uq_gguf_type type, void* wq, uint16_t* scales, int N, int K, void* stream) {
    if (type != UQ_GGUF_Q4_0 && type != UQ_GGUF_Q8_0) return fail(UQ_ERR_UNSUPPORTED, "unknown GGUF block type %d", type);
    if (N < 0 || K < 0) return fail(UQ_ERR_INVALID, "negative size");
    if (K % 32) return fail(UQ_ERR_INVALID, "K=%d is not a multiple of the 32-weight block", K);
    if ((long long)N * K == 0) return UQ_OK;
    if (!blocks || !wq || !scales) return fail(UQ_ERR_INVALID, "null pointer");
    if (!aligned16(wq) || !aligned16(scales)) return fail(UQ_ERR_ALIGN, "wq and scales must be 16-byte aligned");
    cudaError_t e = uq::launch_pack_gguf(type == UQ_GGUF_Q4_0 ? 0 : 1, static_cast<const uint8_t*>(blocks),
                                         static_cast<uint8_t*>(wq), scales, N, K, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? UQ_OK : cuda_fail(e, "GGUF pack launch");
}

namespace {
bool a8_format(int fmt) { return fmt == UQ_INT4_SYM || fmt == UQ_INT4_ASYM || fmt == UQ_INT8_SYM; }
// the shape fields of one A8 GEMV launch over Mb rows (gemv_plan then sets the work split)
void a8_args(uq::GemvArgs& a, const uq::Layout& L, int Mb, int N, int K, int group) {
    a.M = Mb; a.N = N; a.K = K; a.group = group; a.a8 = 1;
    a.NB = L.NB; a.KB = L.KB; a.T = (long long)L.NB * L.KB;
}
}  // namespace

uq_status uq_gemm_w4a8(const uint16_t* x, const void* wq, const void* scales, const void* zeros, uint16_t* y,
                       int M, int N, int K, int group, uq_fmt fmt, void* stream) {
    if (!a8_format(fmt)) return fail(UQ_ERR_UNSUPPORTED, "W4A8 takes INT4_SYM, INT4_ASYM or INT8_SYM weights");
    uq_status s = check_shape(N, K, group, fmt);
    if (s != UQ_OK) return s;
    if (M < 0) return fail(UQ_ERR_INVALID, "negative M");
    if (M == 0 || N == 0) return UQ_OK;
    if (!y) return fail(UQ_ERR_INVALID, "y is NULL");
    if (!aligned16(y)) return fail(UQ_ERR_ALIGN, "y must be 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, (size_t)M * N * 2, st);
        return e == cudaSuccess ? UQ_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (!x || !wq) return fail(UQ_ERR_INVALID, "x or wq is NULL");
    if (!aligned16(x) || !aligned16(wq)) return fail(UQ_ERR_ALIGN, "x and wq must be 16-byte aligned");
    if ((s = check_meta_ptrs(scales, zeros, fmt)) != UQ_OK) return s;
    DeviceState* ds = nullptr;
    int dev = 0;
    if ((s = device_state(&ds, &dev)) != UQ_OK) return s;
    const uq::Layout L(N, K, fmt);
    const int Kp = L.Kp, G = (Kp + group - 1) / group;
    // scratch: x codes [M][Kp] | s_x [M] | per (row, group) code sums [M][G]; partial sums
    const size_t xq_b = ((size_t)M * Kp + 255) / 256 * 256, sx_b = ((size_t)M * 4 + 255) / 256 * 256;
    const size_t aux = xq_b + sx_b + (size_t)M * G * sizeof(int);
    Workspace* ws = nullptr;
    const int rows8 = M < 8 ? M : 8;
    if ((s = workspace(dev, st, (size_t)L.NB * L.KB * RB_ROWS * rows8 * sizeof(float), (size_t)L.NB * sizeof(unsigned int),
                       &ws, aux)) != UQ_OK)
        return s;
    int8_t* xq = reinterpret_cast<int8_t*>(ws->aux);
    float* sx = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws->aux) + xq_b);
    int* sxl = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ws->aux) + xq_b + sx_b);
    cudaError_t e = uq::launch_quant_x(x, xq, sx, sxl, M, K, Kp, group, fmt == UQ_INT8_SYM ? 0 : 1, st);
    if (e != cudaSuccess) return cuda_fail(e, "activation quantization launch");
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mb = (M - m0) < 8 ? (M - m0) : 8;
        uq::GemvArgs a = {};
        a8_args(a, L, mb, N, K, group);
        a.x = x;
        a.wq = static_cast<const uint8_t*>(wq);
        a.scales = static_cast<const uint8_t*>(scales);
        a.zc = static_cast<const uint8_t*>(zeros);
        a.y = y + (long long)m0 * N;
        a.ldx = K; a.ldy = N;
        a.partials = ws->partials;
        a.tickets = ws->tickets;
        a.fault = ds->words;
        const int grid = uq::gemv_plan(a, fmt, ds->sms);
        e = uq::launch_gemv_a8(fmt, a, xq + (long long)m0 * Kp, sx + m0, sxl + (long long)m0 * G, Kp, grid, st);
        if (e != cudaSuccess) return cuda_fail(e, "W4A8 GEMV launch");
    }
    return UQ_OK;
}

uq_status uq_gemm_w4a8_kernel_count(int M, int N, int K, int group, uq_fmt fmt, int* count) {
    if (!count) return fail(UQ_ERR_INVALID, "null pointer");
    *count = 0;
    if (!a8_format(fmt)) return fail(UQ_ERR_UNSUPPORTED, "W4A8 takes INT4_SYM, INT4_ASYM or INT8_SYM weights");
    uq_status s = check_shape(N, K, group, fmt);
    if (s != UQ_OK) return s;
    if (M < 0) return fail(UQ_ERR_INVALID, "negative M");
    if (M == 0 || N == 0) return UQ_OK;
    if (K == 0) { *count = 1; return UQ_OK; }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms < 1) return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidDevice, "SM count");
    const uq::Layout L(N, K, fmt);
    int n = (M + 65534) / 65535;                                 // the activation quantization (65535 rows a launch)
    for (int m0 = 0; m0 < M; m0 += 8) {
        uq::GemvArgs a = {};
        a8_args(a, L, (M - m0) < 8 ? (M - m0) : 8, N, K, group);
        uq::gemv_plan(a, fmt, sms);
        n += uq::gemv_launches(fmt, a);
    }
    *count = n;
    return UQ_OK;
}

uq_status uq_unpack_codes(const void* wq, int8_t* codes, int N, int K, int group, uq_fmt fmt, void* stream) {
    uq_status s = check_shape(N, K, group, fmt);
    if (s != UQ_OK) return s;
    if ((long long)N * K == 0) return UQ_OK;
    if (!wq || !codes) return fail(UQ_ERR_INVALID, "null pointer");
    if (!aligned16(wq) || !aligned16(codes)) return fail(UQ_ERR_ALIGN, "pointers must be 16-byte aligned");
    cudaError_t e = uq::launch_unpack(fmt, static_cast<const uint8_t*>(wq), codes, N, K,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "unpack launch");
    return UQ_OK;
}

uq_status uq_dequant(const void* wq, const void* scales, const void* zeros_or_codebook, float* w, int N, int K,
                     int group, uq_fmt fmt, void* stream) {
    uq_status s = check_shape(N, K, group, fmt);
    if (s != UQ_OK) return s;
    if ((long long)N * K == 0) return UQ_OK;
    if (!wq || !w) return fail(UQ_ERR_INVALID, "null pointer");
    if (!aligned16(wq) || !aligned16(w)) return fail(UQ_ERR_ALIGN, "pointers must be 16-byte aligned");
    if ((s = check_meta_ptrs(scales, zeros_or_codebook, fmt)) != UQ_OK) return s;
    cudaError_t e = uq::launch_dequant(fmt, static_cast<const uint8_t*>(wq), static_cast<const uint8_t*>(scales),
                                       static_cast<const uint8_t*>(zeros_or_codebook), w, N, K, group,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dequant launch");
    return UQ_OK;
}

uq_status uq_quantize(const float* w, int8_t* codes, uint16_t* scales, void* zeros, const float* codebook, int N,
                      int K, int group, uq_fmt fmt, void* stream) {
    if (fmt == UQ_K4) return fail(UQ_ERR_INVALID, "use uq_quantize_k4 for UQ_K4");
    uq_status s = check_shape(N, K, group, fmt);
    if (s != UQ_OK) return s;
    if ((long long)N * K == 0) return UQ_OK;
    if (!w || !codes || !scales) return fail(UQ_ERR_INVALID, "null pointer");
    const bool wants_z = (fmt == UQ_INT4_ASYM || fmt == UQ_INT2_ASYM);
    if (wants_z != (zeros != nullptr)) return fail(UQ_ERR_INVALID, "zeros must be given exactly for the ASYM formats");
    if ((fmt == UQ_NF4) != (codebook != nullptr)) return fail(UQ_ERR_INVALID, "codebook must be given exactly for UQ_NF4");
    if (!aligned16(w) || !aligned16(codes) || !aligned16(scales) || (zeros && !aligned16(zeros)) ||
        (codebook && !aligned16(codebook)))
        return fail(UQ_ERR_ALIGN, "pointers must be 16-byte aligned");
    cudaError_t e = uq::launch_quantize(fmt, w, codes, scales, zeros, codebook, N, K, group,
                                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    return UQ_OK;
}

uq_status uq_quantize_k4(const float* w, int8_t* codes, uint16_t* d, uint16_t* dmin, uint8_t* sc, uint8_t* m,
                         int N, int K, void* stream) {
    uq_status s = check_shape(N, K, 256, UQ_K4);
    if (s != UQ_OK) return s;
    if ((long long)N * K == 0) return UQ_OK;
    if (!w || !codes || !d || !dmin || !sc || !m) return fail(UQ_ERR_INVALID, "null pointer");
    if (!aligned16(w) || !aligned16(codes) || !aligned16(d) || !aligned16(dmin) || !aligned16(sc) || !aligned16(m))
        return fail(UQ_ERR_ALIGN, "pointers must be 16-byte aligned");
    cudaError_t e = uq::launch_quantize_k4(w, codes, d, dmin, sc, m, N, K, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "quantize_k4 launch");
    return UQ_OK;
}

uq_status uq_set_gemm_path(int path) {
    if (path < 0 || path > 2)
        return fail(UQ_ERR_INVALID, "path must be 0 (automatic), 1 (tensor cores) or 2 (mma.sync GEMM)");
    g_path.store(path);
    return UQ_OK;
}

uq_status uq_set_launch_overlap(int enable) {
    uq::g_overlap.store(enable ? 1 : 0);
    return UQ_OK;
}

uq_status uq_gemm_kernel_count(int M, int N, int K, int group, uq_fmt fmt, int* count) {
    if (!count) return fail(UQ_ERR_INVALID, "null pointer");
    *count = 0;
    uq_status s = check_shape(N, K, group, fmt);
    if (s != UQ_OK) return s;
    if (M < 0) return fail(UQ_ERR_INVALID, "negative M");
    if (M == 0 || N == 0) return UQ_OK;
    if (K == 0) { *count = 1; return UQ_OK; }                          // the cudaMemsetAsync of y
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms < 1) return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidDevice, "SM count");
    int n = 0;
    const Route rt = route(fmt, M, N, K);
    if (rt == ROUTE_MMA_GEMM) {
        // per block of at most 64 rows: the mma.sync GEMM (K4: after its x column-sum pre-kernel;
        // plus the second pass when its k range is split); a last block of at most 8 rows: the GEMV
        const uq::Layout L(N, K, fmt);
        for (int m0 = 0; m0 < M; m0 += 64) {
            const int mb = (M - m0) < 64 ? (M - m0) : 64;
            if (mb > 8) {
                n += gemm_mma_launches(fmt, mb, N, K, sms);
            } else {
                uq::GemvArgs a = {};
                a.M = mb; a.N = N; a.K = K; a.group = group;
                a.NB = L.NB; a.KB = L.KB; a.T = (long long)L.NB * L.KB;
                uq::gemv_plan(a, fmt, sms);
                n += uq::gemv_launches(fmt, a);
            }
        }
    } else if (rt == ROUTE_TC) {
        // per block of at most 64 rows: the GEMM (K4: after its x column-sum pre-kernel)
        for (int m0 = 0; m0 < M; m0 += 64) n += (fmt == UQ_K4) ? 2 : 1;
    } else {
        // per block of at most 8 rows: one GEMV launch
        const uq::Layout L(N, K, fmt);
        for (int m0 = 0; m0 < M; m0 += 8) {
            const int mb = (M - m0) < 8 ? (M - m0) : 8;
            uq::GemvArgs a = {};
            a.M = mb; a.N = N; a.K = K; a.group = group;
            a.NB = L.NB; a.KB = L.KB; a.T = (long long)L.NB * L.KB;
            uq::gemv_plan(a, fmt, sms);
            n += uq::gemv_launches(fmt, a);
        }
    }
    *count = n;
    return UQ_OK;
}

uq_status uq_device_fault(unsigned int* flag) {
    if (!flag) return fail(UQ_ERR_INVALID, "null pointer");
    *flag = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    // the word of uq_gemm and the debug calls (only if this device has run one: nothing is allocated here)
    unsigned int v = 0;
    unsigned int* words = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_dev.find(dev);
        if (it != g_dev.end()) words = it->second.words;
    }
    if (words) {
        e = cudaMemcpy(&v, words, sizeof v, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
        if (v) {
            // a kernel returned early: its tickets may be left non-zero; clear this device's workspaces
            cudaMemset(words, 0, sizeof v);
            std::lock_guard<std::mutex> lk(g_mu);
            for (auto& kv : g_ws)
                if (kv.first.first == dev && kv.second.tickets)
                    cudaMemset(kv.second.tickets, 0, kv.second.ticket_bytes);
            for (auto& r : g_retired)
                if (r.dev == dev && r.tickets) cudaMemset(r.ptr, 0, r.bytes);
        }
    }
    // the word of uq_gemm_noalloc (the first word of its static array)
    unsigned int vn = 0;
    e = uq::noalloc_take_fault(&vn);
    if (e != cudaSuccess) return cuda_fail(e, "reading the no-alloc fault word");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    *flag = v | vn;
    return UQ_OK;
}

}  // extern "C"
