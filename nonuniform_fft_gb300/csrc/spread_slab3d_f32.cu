// 3D single-precision slab spreader (spread_slab3d.cuh): launcher and bins.
#include "spread_slab3d.cuh"

namespace nufft {

bool slab3d_supported(int w, int dtype) { return dtype == 0 && w >= 2 && w <= kSlab3DMaxWidth; }

// Bins one window origin thick in z, 33 - w origins wide (lane L owns padded
// column L: w - 1 columns of padding), 32 rows (rows only slide the register
// windows; measured on the 3D single-precision workload at w = 7 with one
// subproblem per bin and cell binning: 4, 8, 12, 16, 24, 32, 48 rows gave
// 5.61, 5.13, 4.99, 4.91, 4.87, 4.84, 4.96 ms).
void slab3d_bins(int w, int *m1, int *m2, int *m3) {
  *m1 = 33 - w;
  *m2 = 32;
  *m3 = 1;
}

cudaError_t launch_spread_slab3d(const nufft_plan_s *p, const void *c) {
  switch (p->w) {
    case 2: return spread_slab3d_w<2>(p, c);
    case 3: return spread_slab3d_w<3>(p, c);
    case 4: return spread_slab3d_w<4>(p, c);
    case 5: return spread_slab3d_w<5>(p, c);
    case 6: return spread_slab3d_w<6>(p, c);
    case 7: return spread_slab3d_w<7>(p, c);
    case 8: return spread_slab3d_w<8>(p, c);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nufft
