// uq_tc_int8s.cu -- instantiates the tensor-core path for UQ_INT8_SYM (one translation unit per format so the
// library builds in parallel).
#include "uq_tc.cuh"

namespace uq {
template cudaError_t launch_tc_fmt<UQ_INT8_SYM>(const CUtensorMap&, const TcArgs&, size_t, int, cudaStream_t);
}  // namespace uq
