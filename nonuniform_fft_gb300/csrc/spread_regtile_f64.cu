// Register-tile 2D spreader instantiated for double precision.
#include "spread_regtile.cuh"

namespace nufft {
template cudaError_t launch_spread_regtile2d<double>(const nufft_plan_s *, const void *);
}  // namespace nufft
