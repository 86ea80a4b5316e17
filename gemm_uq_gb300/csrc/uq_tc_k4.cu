// uq_tc_k4.cu -- instantiates the tensor-core path for UQ_K4 (one translation unit per format so the
// library builds in parallel).
#include "uq_tc.cuh"

namespace uq {
template cudaError_t launch_tc_fmt<UQ_K4>(const CUtensorMap&, const TcArgs&, size_t, int, cudaStream_t);
}  // namespace uq
