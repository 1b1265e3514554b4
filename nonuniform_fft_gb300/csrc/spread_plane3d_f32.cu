// Register-tile 3D spreader instantiated for float precision.
#include "spread_plane3d.cuh"

namespace nufft {
template cudaError_t launch_spread_plane3d<float>(const nufft_plan_s *, const void *);

// Bin size of the 3D register-tile spreader (see Plane3DChoice).
void plane3d_bins(int w, int dtype, int *m1, int *m2, int *m3) {
  // rows per bin (free in the kernel): 8 in single precision, 4 in double
  // (option sweeps of the 3D workloads: 8 rows best at w = 7 in single
  // precision; 4 rows with M_sub 2048 best at w = 13 in double, 93.7 against
  // 98.8 ms for 16 rows with M_sub 8192)
  if (dtype == 0) {
    plane3d_bins_t<float>(w, m1, m3);
    *m2 = 8;
  } else {
    plane3d_bins_t<double>(w, m1, m3);
    *m2 = 4;
  }
}
}  // namespace nufft
