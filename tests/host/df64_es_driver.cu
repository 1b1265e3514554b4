// Host driver for the accuracy test of the two-float ES kernel in
// nonuniform_fft_gb300/csrc/df64.cuh (compiled as host code).  Reads lines
// "z beta" from stdin and prints phi as hi and lo.
#include <cstdio>

#include "../../nonuniform_fft_gb300/csrc/df64.cuh"

int main() {
  double z, beta;
  while (std::scanf("%lf %lf", &z, &beta) == 2) {
    const nufft::DF r = nufft::df_es_kernel(nufft::df_from(z), nufft::df_from(beta));
    std::printf("%.17g %.17g\n", (double)r.hi, (double)r.lo);
  }
  return 0;
}
