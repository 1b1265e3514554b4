// Register-tile 2D spreader instantiated for float precision.
#include "spread_regtile.cuh"

namespace nufft {
template cudaError_t launch_spread_regtile2d<float>(const nufft_plan_s *, const void *);

// Bin size of the register-tile spreader: 32 C - 2 ceil(w/2) cells wide
// (C tile columns per lane), so the padded bin has 32 C columns; 32 rows (the
// rows only cost a sliding window of registers; in the option sweeps 32 rows
// matched 64 on uniform points and beat them by 5 % on clustered ones).
void regtile2d_bins(int w, int cols, int *m1, int *m2) {
  const int pad = (w + 1) / 2;
  *m1 = 32 * cols - 2 * pad;
  *m2 = 32;
}
}  // namespace nufft
