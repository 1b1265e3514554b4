// Spreading / interpolation kernels instantiated for 3D, float precision.
#include "spreadinterp.cuh"

namespace nufft {
template cudaError_t launch_spread_t<3, float>(const nufft_plan_s *, const void *);
template cudaError_t launch_interp_t<3, float>(const nufft_plan_s *, void *);
}  // namespace nufft
