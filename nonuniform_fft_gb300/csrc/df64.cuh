// Double-single ("two-float") arithmetic for the double-precision kernels.
//
// A value is an unevaluated sum hi + lo of two floats with |lo| <= ulp(hi)/2,
// about 48 significant bits.  The operations are the error-free
// transformations of Dekker (1971, "A floating-point technique for extending
// the available precision") and Knuth's two-sum, built from single-precision
// adds, multiplies and fused multiply-adds.  This part executes about 64
// single-precision FMAs per double-precision FMA, so the w^d
// multiply-accumulates per point of the double-precision spreading and
// interpolation run in this form, and so can the kernel values themselves
// (df_es_kernel).  Every operation uses the _rn intrinsics so the compiler
// cannot contract or reorder the error terms.
#pragma once

#include <cuda_runtime.h>

#ifndef __CUDA_ARCH__
#include <cmath>
#endif

namespace nufft {

// Single-precision operations that the compiler may not fuse or reorder: the
// _rn intrinsics on the device; on the host (where the same code is compiled
// for its accuracy test) plain operations, built with contraction off.
#ifdef __CUDA_ARCH__
#define DF_ADD(a, b) __fadd_rn(a, b)
#define DF_SUB(a, b) __fsub_rn(a, b)
#define DF_MUL(a, b) __fmul_rn(a, b)
#define DF_FMA(a, b, c) __fmaf_rn(a, b, c)
#define DF_SQRT(a) __fsqrt_rn(a)
#define DF_DIV(a, b) __fdiv_rn(a, b)
#define DF_D2F(x) __double2float_rn(x)
#define DF_DSUB(a, b) __dsub_rn(a, b)
#define DF_DADD(a, b) __dadd_rn(a, b)
#else
#define DF_ADD(a, b) ((float)((a) + (b)))
#define DF_SUB(a, b) ((float)((a) - (b)))
#define DF_MUL(a, b) ((float)((a) * (b)))
#define DF_FMA(a, b, c) std::fmaf(a, b, c)
#define DF_SQRT(a) std::sqrt((float)(a))
#define DF_DIV(a, b) ((float)((a) / (b)))
#define DF_D2F(x) ((float)(x))
#define DF_DSUB(a, b) ((a) - (b))
#define DF_DADD(a, b) ((a) + (b))
#endif
#define DF_HD __host__ __device__ __forceinline__

struct DF {
  float hi, lo;
};

// Nearest two-float to a double (exact up to the 48-bit precision).
DF_HD DF df_from(double x) {
  const float h = DF_D2F(x);
  DF r;
  r.hi = h;
  r.lo = DF_D2F(DF_DSUB(x, (double)h));
  return r;
}

DF_HD double df_to(DF a) { return DF_DADD((double)a.hi, (double)a.lo); }

// Renormalise s + e into a two-float (requires |s| >= |e| or s == 0).
DF_HD DF df_quick(float s, float e) {
  const float h = DF_ADD(s, e);
  DF r;
  r.hi = h;
  r.lo = DF_SUB(e, DF_SUB(h, s));
  return r;
}

// a * b.
DF_HD DF df_mul(DF a, DF b) {
  const float p = DF_MUL(a.hi, b.hi);
  float e = DF_FMA(a.hi, b.hi, -p);       // exact error of the leading product
  e = DF_FMA(a.hi, b.lo, e);
  e = DF_FMA(a.lo, b.hi, e);
  return df_quick(p, e);
}

// acc += a * b.
DF_HD void df_fma(DF &acc, DF a, DF b) {
  const float p = DF_MUL(a.hi, b.hi);
  float pe = DF_FMA(a.hi, b.hi, -p);
  pe = DF_FMA(a.hi, b.lo, pe);
  pe = DF_FMA(a.lo, b.hi, pe);
  // two-sum of acc.hi and p
  const float s = DF_ADD(acc.hi, p);
  const float v = DF_SUB(s, acc.hi);
  float e = DF_ADD(DF_SUB(acc.hi, DF_SUB(s, v)), DF_SUB(p, v));
  e = DF_ADD(e, DF_ADD(acc.lo, pe));
  acc = df_quick(s, e);
}

// acc += a * b without renormalising: acc.hi takes the float sum, and the
// exact TwoSum error of that addition plus the product's own error terms go
// to acc.lo in float arithmetic, so acc.hi + acc.lo carries the running sum
// while |acc.lo| grows by at most one unit in the last place of acc.hi per
// step.  After n steps the float rounding of acc.lo is below n^2 2^-48 of
// the largest partial sum; callers renormalise (df_sum) after a short run,
// at most 16 terms.
DF_HD void df_fma_lazy(DF &acc, DF a, DF b) {
  const float p = DF_MUL(a.hi, b.hi);
  float pe = DF_FMA(a.hi, b.hi, -p);
  pe = DF_FMA(a.hi, b.lo, pe);
  pe = DF_FMA(a.lo, b.hi, pe);
  const float s = DF_ADD(acc.hi, p);
  const float v = DF_SUB(s, acc.hi);
  const float e = DF_ADD(DF_SUB(acc.hi, DF_SUB(s, v)), DF_SUB(p, v));
  acc.hi = s;
  acc.lo = DF_ADD(acc.lo, DF_ADD(e, pe));
}

// a + b.
DF_HD DF df_sum(DF a, DF b) {
  const float s = DF_ADD(a.hi, b.hi);
  const float v = DF_SUB(s, a.hi);
  float e = DF_ADD(DF_SUB(a.hi, DF_SUB(s, v)), DF_SUB(b.hi, v));
  e = DF_ADD(e, DF_ADD(a.lo, b.lo));
  return df_quick(s, e);
}

DF_HD DF df_neg(DF a) { return DF{-a.hi, -a.lo}; }

// a / b (b > 0): one correction of the single-precision quotient.
DF_HD DF df_div(DF a, DF b) {
  const float q0 = DF_DIV(a.hi, b.hi);
  const DF r = df_sum(a, df_neg(df_mul(DF{q0, 0.f}, b)));
  const float q1 = DF_DIV(r.hi, b.hi);
  return df_quick(q0, q1);
}

// sqrt(a) for a >= 0: one Newton correction of the single-precision root,
// s = s0 + (a - s0^2) / (2 s0).
DF_HD DF df_sqrt(DF a) {
  if (!(a.hi > 0.f)) return DF{0.f, 0.f};
  const float s0 = DF_SQRT(a.hi);
  const DF r = df_sum(a, df_neg(df_mul(DF{s0, 0.f}, DF{s0, 0.f})));
  return df_quick(s0, DF_DIV(r.hi, DF_MUL(2.f, s0)));
}

// exp(a) for -88 < a <= 0.  Cody-Waite reduction a = k ln2 + r with ln2
// split into three floats (k ln2 exact in the first two parts for |k| < 128,
// the first part having 16 significant bits), |r| <= ln2 / 2; e^r by its
// Taylor series to degree 13 (truncation below 1e-17 on that interval);
// then e^a = 2^k e^r.
DF_HD DF df_exp(DF a) {
  constexpr double LN2 = 0.693147180559945309417232121458176568;
  constexpr float C1 = 0.693145751953125f;                       // 16 bits
  constexpr float C2 = (float)(LN2 - (double)C1);
  constexpr float C3 = (float)(LN2 - (double)C1 - (double)C2);
  const float kf = rintf(DF_MUL(a.hi, 1.44269504088896340736f));
  DF r = df_sum(a, DF{DF_MUL(-kf, C1), 0.f});    // exact product
  r = df_sum(r, df_neg(df_mul(DF{kf, 0.f}, DF{C2, 0.f})));
  r = df_sum(r, df_neg(df_mul(DF{kf, 0.f}, DF{C3, 0.f})));
  // Horner: sum_{n=0}^{13} r^n / n!
  constexpr double F[14] = {1.0, 1.0, 1.0 / 2, 1.0 / 6, 1.0 / 24, 1.0 / 120, 1.0 / 720, 1.0 / 5040,
                            1.0 / 40320, 1.0 / 362880, 1.0 / 3628800, 1.0 / 39916800,
                            1.0 / 479001600, 1.0 / 6227020800.0};
  DF p{(float)F[13], (float)(F[13] - (double)(float)F[13])};
#pragma unroll
  for (int n = 12; n >= 0; n--) {
    const DF c{(float)F[n], (float)(F[n] - (double)(float)F[n])};
    p = df_sum(df_mul(p, r), c);
  }
  const int k = (int)kf;
  return DF{ldexpf(p.hi, k), ldexpf(p.lo, k)};
}

// A table of 2^(j/64), j = 0..63, shortens the series: a = (64 k + j) ln2/64
// + r with |r| <= ln2/128 (Cody-Waite with ln2/64 split in three floats, the
// first with 11 significant bits so that n times it is exact for |n| < 2^13),
// e^r by its Taylor series to degree 6 (truncation below 3e-20), then e^a =
// 2^k 2^(j/64) e^r.  The table entries come from df_exp of the arguments
// j ln2/64, formed from the same split (df_exp2_64).
constexpr double kLn2Over64 = 0.693147180559945309417232121458176568 / 64;
constexpr float kL64a = 0.010833740234375f;  // 1420 / 2^17
constexpr float kL64b = (float)(kLn2Over64 - (double)kL64a);
constexpr float kL64c = (float)(kLn2Over64 - (double)kL64a - (double)kL64b);

DF_HD DF df_exp2_64(int j) {
  const float jf = (float)j;
  DF arg{DF_MUL(jf, kL64a), 0.f};  // exact: 6 + 11 bits
  arg = df_sum(arg, df_mul(DF{jf, 0.f}, DF{kL64b, 0.f}));
  arg = df_sum(arg, df_mul(DF{jf, 0.f}, DF{kL64c, 0.f}));
  return df_exp(arg);
}

DF_HD DF df_exp_tab(DF a, const DF *tab) {
  const float nf = rintf(DF_MUL(a.hi, 92.33248261689366f));  // 64 / ln2
  DF r = df_sum(a, DF{DF_MUL(-nf, kL64a), 0.f});             // exact product
  r = df_sum(r, df_neg(df_mul(DF{nf, 0.f}, DF{kL64b, 0.f})));
  r = df_sum(r, df_neg(df_mul(DF{nf, 0.f}, DF{kL64c, 0.f})));
  constexpr double F[7] = {1.0, 1.0, 1.0 / 2, 1.0 / 6, 1.0 / 24, 1.0 / 120, 1.0 / 720};
  DF p{(float)F[6], (float)(F[6] - (double)(float)F[6])};
#pragma unroll
  for (int n = 5; n >= 0; n--) {
    const DF c{(float)F[n], (float)(F[n] - (double)(float)F[n])};
    p = df_sum(df_mul(p, r), c);
  }
  const int n = (int)nf;
  p = df_mul(p, tab[n & 63]);  // n = 64 (n >> 6) + (n & 63)
  const int k = n >> 6;
  return DF{ldexpf(p.hi, k), ldexpf(p.lo, k)};
}

// The ES kernel phi(z) = exp(beta (sqrt(1 - z^2) - 1)) (eq. (5)) for |z| <= 1,
// with the exponent written -beta z^2 / (1 + sqrt(1 - z^2)) so that nothing
// cancels near z = 0, and 1 - z^2 as (1 - z)(1 + z) so that nothing cancels
// near |z| = 1.
DF_HD DF df_es_kernel(DF z, DF beta) {
  const DF one{1.f, 0.f};
  const DF om = df_mul(df_sum(one, df_neg(z)), df_sum(one, z));
  const DF s = df_sqrt(om);
  const DF z2 = df_mul(z, z);
  const DF ex = df_neg(df_mul(beta, df_div(z2, df_sum(one, s))));
  return df_exp(ex);
}

// The same with the table exponential (tab: the 64 values of df_exp2_64).
DF_HD DF df_es_kernel(DF z, DF beta, const DF *tab) {
  const DF one{1.f, 0.f};
  const DF om = df_mul(df_sum(one, df_neg(z)), df_sum(one, z));
  const DF s = df_sqrt(om);
  const DF z2 = df_mul(z, z);
  const DF ex = df_neg(df_mul(beta, df_div(z2, df_sum(one, s))));
  return df_exp_tab(ex, tab);
}

}  // namespace nufft
