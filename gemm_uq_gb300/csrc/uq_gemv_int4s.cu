// uq_gemv_int4s.cu -- instantiates the small-M GEMV for UQ_INT4_SYM (one translation unit per format
// so the library builds in parallel).
#include "uq_gemv.cuh"

namespace uq {
template cudaError_t launch_gemv_fmt<UQ_INT4_SYM>(const GemvArgs&, int, cudaStream_t);
}  // namespace uq
