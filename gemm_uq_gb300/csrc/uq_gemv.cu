// uq_gemv.cu -- dispatch of the small-M GEMV over formats (kernels instantiated in uq_gemv_*.cu).
#include "uq_gemv.cuh"

namespace uq {

extern template cudaError_t launch_gemv_fmt<UQ_INT4_SYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_INT4_ASYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_INT8_SYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_INT2_ASYM>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_NF4>(const GemvArgs&, int, cudaStream_t);
extern template cudaError_t launch_gemv_fmt<UQ_K4>(const GemvArgs&, int, cudaStream_t);

size_t gemv_smem_bytes(int fmt, int K, int group, int M) { return gemv_smem_bytes_impl(fmt, K, group, M); }
int gemv_warps(int fmt) { return gemv_warps_impl(fmt); }
int gemv_grid(int fmt, int P, int sms) {
    // the mma kernel strides its workers over the CTAs, so it can use every SM whatever P is
    if (gemv_is_mma(fmt)) return P < sms ? P : sms;
    return (P + GEMV_WARPS - 1) / GEMV_WARPS;
}
size_t gemv_partials_floats(int P, int M) { return gemv_partials_floats_impl(P, M); }

cudaError_t launch_gemv(int fmt, const GemvArgs& a, int grid, cudaStream_t st) {
    switch (fmt) {
        case UQ_INT4_SYM: return launch_gemv_fmt<UQ_INT4_SYM>(a, grid, st);
        case UQ_INT4_ASYM: return launch_gemv_fmt<UQ_INT4_ASYM>(a, grid, st);
        case UQ_INT8_SYM: return launch_gemv_fmt<UQ_INT8_SYM>(a, grid, st);
        case UQ_INT2_ASYM: return launch_gemv_fmt<UQ_INT2_ASYM>(a, grid, st);
        case UQ_NF4: return launch_gemv_fmt<UQ_NF4>(a, grid, st);
        case UQ_K4: return launch_gemv_fmt<UQ_K4>(a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace uq
