// Stand-ins for the per-format GEMV launchers, so the planner's translation unit links without the
// kernels (gemv_plan_probe.cu never launches anything).  Full specializations carry the same symbol
// names as the library's instantiations.
#include <cuda_runtime.h>

namespace uq {
struct GemvArgs;
template <int FMT>
cudaError_t launch_gemv_fmt(const GemvArgs&, int, cudaStream_t);
template <> cudaError_t launch_gemv_fmt<0>(const GemvArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
template <> cudaError_t launch_gemv_fmt<1>(const GemvArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
template <> cudaError_t launch_gemv_fmt<2>(const GemvArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
template <> cudaError_t launch_gemv_fmt<3>(const GemvArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
template <> cudaError_t launch_gemv_fmt<4>(const GemvArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
template <> cudaError_t launch_gemv_fmt<5>(const GemvArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace uq
