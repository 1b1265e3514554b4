// Host driver for the accuracy test of the two-float ES kernel in
// nonuniform_fft_gb300/csrc/df64.cuh (compiled as host code).  Reads lines
// "z beta" from stdin and prints phi as hi and lo, first by the series
// exponential (df_es_kernel) and then by the table exponential with the
// table of 2^(j/64) built as the kernels build it (df_exp2_64).
#include <cstdio>

#include "../../nonuniform_fft_gb300/csrc/df64.cuh"

int main() {
  nufft::DF tab[64];
  for (int j = 0; j < 64; j++) tab[j] = nufft::df_exp2_64(j);
  double z, beta;
  while (std::scanf("%lf %lf", &z, &beta) == 2) {
    const nufft::DF zd = nufft::df_from(z), bd = nufft::df_from(beta);
    const nufft::DF r = nufft::df_es_kernel(zd, bd);
    const nufft::DF t = nufft::df_es_kernel(zd, bd, tab);
    std::printf("%.17g %.17g %.17g %.17g\n", (double)r.hi, (double)r.lo, (double)t.hi, (double)t.lo);
  }
  return 0;
}
