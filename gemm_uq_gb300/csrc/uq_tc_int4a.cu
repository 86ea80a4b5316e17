// uq_tc_int4a.cu -- instantiates the tensor-core path for UQ_INT4_ASYM (one translation unit per format so the
// library builds in parallel).
#include "uq_tc.cuh"

namespace uq {
template cudaError_t launch_tc_fmt<UQ_INT4_ASYM>(const CUtensorMap&, const TcArgs&, size_t, int, cudaStream_t);
}  // namespace uq
