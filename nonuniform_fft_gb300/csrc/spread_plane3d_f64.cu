// Register-tile 3D spreader instantiated for double precision.
#include "spread_plane3d.cuh"

namespace nufft {
template cudaError_t launch_spread_plane3d<double>(const nufft_plan_s *, const void *);
}  // namespace nufft
