// uq_gemv_nf4.cu -- instantiates the small-M GEMV for UQ_NF4 (one translation unit per format
// so the library builds in parallel).
#include "uq_gemv.cuh"

namespace uq {
template cudaError_t launch_gemv_fmt<UQ_NF4>(const GemvArgs&, int, cudaStream_t);
}  // namespace uq
