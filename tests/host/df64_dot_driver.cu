// Host driver for the accuracy test of the two-float dot products in
// nonuniform_fft_gb300/csrc/df64.cuh (compiled as host code).  Each input
// line is "n a_1 b_1 ... a_n b_n" (doubles); the driver splits every value
// into a two-float, accumulates the products with df_fma_lazy in two
// interleaved chains (odd and even terms, as the double-precision
// interpolator does) and with df_fma in one chain, and prints both sums as
// "hi lo hi lo".
#include <cstdio>

#include "../../nonuniform_fft_gb300/csrc/df64.cuh"

int main() {
  int n;
  while (std::scanf("%d", &n) == 1) {
    nufft::DF s0{0.f, 0.f}, s1{0.f, 0.f}, s{0.f, 0.f};
    for (int i = 0; i < n; i++) {
      double a, b;
      if (std::scanf("%lf %lf", &a, &b) != 2) return 1;
      const nufft::DF da = nufft::df_from(a), db = nufft::df_from(b);
      nufft::df_fma_lazy(i % 2 == 0 ? s0 : s1, da, db);
      nufft::df_fma(s, da, db);
    }
    const nufft::DF lazy = nufft::df_sum(s0, s1);
    std::printf("%.17g %.17g %.17g %.17g\n", (double)lazy.hi, (double)lazy.lo, (double)s.hi, (double)s.lo);
  }
  return 0;
}
