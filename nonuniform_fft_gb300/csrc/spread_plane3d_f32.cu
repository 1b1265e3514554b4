// Register-tile 3D spreader instantiated for float precision.
#include "spread_plane3d.cuh"

namespace nufft {
template cudaError_t launch_spread_plane3d<float>(const nufft_plan_s *, const void *);

// Bin size of the 3D register-tile spreader (see Plane3DChoice).
void plane3d_bins(int w, int dtype, int *m1, int *m2, int *m3) {
  // rows per bin (free in the kernel): 8 in single precision, 16 in double
  // (measured on the 3D workloads: 6.59 against 6.72 ms, 98.5 against 99.7 ms)
  if (dtype == 0) {
    plane3d_bins_t<float>(w, m1, m3);
    *m2 = 8;
  } else {
    plane3d_bins_t<double>(w, m1, m3);
    *m2 = 16;
  }
}
}  // namespace nufft
