// Spreading / interpolation kernels instantiated for 2D, float precision.
#include "spreadinterp.cuh"

namespace nufft {
template cudaError_t launch_spread_t<2, float>(const nufft_plan_s *, const void *);
template cudaError_t launch_interp_t<2, float>(const nufft_plan_s *, void *);

}  // namespace nufft
