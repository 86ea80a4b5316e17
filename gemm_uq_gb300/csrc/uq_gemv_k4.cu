// uq_gemv_k4.cu -- instantiates the small-M GEMV for UQ_K4 (one translation unit per format
// so the library builds in parallel).
#include "uq_gemv.cuh"

namespace uq {
template cudaError_t launch_gemv_fmt<UQ_K4>(const GemvArgs&, int, cudaStream_t);
}  // namespace uq
