// Double-single ("two-float") arithmetic for the double-precision kernels.
//
// A value is an unevaluated sum hi + lo of two floats with |lo| <= ulp(hi)/2,
// about 48 significant bits.  The operations are the error-free
// transformations of Dekker (1971, "A floating-point technique for extending
// the available precision") and Knuth's two-sum, built from single-precision
// adds, multiplies and fused multiply-adds.  This part executes about 64
// single-precision FMAs per double-precision FMA, so the w^d
// multiply-accumulates per point of the double-precision spreading and
// interpolation run in this form, while the kernel values themselves are
// evaluated in double.  Every operation uses the _rn intrinsics so the
// compiler cannot contract or reorder the error terms.
#pragma once

#include <cuda_runtime.h>

namespace nufft {

struct DF {
  float hi, lo;
};

// Nearest two-float to a double (exact up to the 48-bit precision).
__device__ __forceinline__ DF df_from(double x) {
  const float h = __double2float_rn(x);
  DF r;
  r.hi = h;
  r.lo = __double2float_rn(__dsub_rn(x, (double)h));
  return r;
}

__device__ __forceinline__ double df_to(DF a) { return __dadd_rn((double)a.hi, (double)a.lo); }

// Renormalise s + e into a two-float (requires |s| >= |e| or s == 0).
__device__ __forceinline__ DF df_quick(float s, float e) {
  const float h = __fadd_rn(s, e);
  DF r;
  r.hi = h;
  r.lo = __fsub_rn(e, __fsub_rn(h, s));
  return r;
}

// a * b.
__device__ __forceinline__ DF df_mul(DF a, DF b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = __fmaf_rn(a.hi, b.hi, -p);       // exact error of the leading product
  e = __fmaf_rn(a.hi, b.lo, e);
  e = __fmaf_rn(a.lo, b.hi, e);
  return df_quick(p, e);
}

// acc += a * b.
__device__ __forceinline__ void df_fma(DF &acc, DF a, DF b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float pe = __fmaf_rn(a.hi, b.hi, -p);
  pe = __fmaf_rn(a.hi, b.lo, pe);
  pe = __fmaf_rn(a.lo, b.hi, pe);
  // two-sum of acc.hi and p
  const float s = __fadd_rn(acc.hi, p);
  const float v = __fsub_rn(s, acc.hi);
  float e = __fadd_rn(__fsub_rn(acc.hi, __fsub_rn(s, v)), __fsub_rn(p, v));
  e = __fadd_rn(e, __fadd_rn(acc.lo, pe));
  acc = df_quick(s, e);
}

// acc += b (two-float plus two-float).
__device__ __forceinline__ void df_add(DF &acc, DF b) {
  const float s = __fadd_rn(acc.hi, b.hi);
  const float v = __fsub_rn(s, acc.hi);
  float e = __fadd_rn(__fsub_rn(acc.hi, __fsub_rn(s, v)), __fsub_rn(b.hi, v));
  e = __fadd_rn(e, __fadd_rn(acc.lo, b.lo));
  acc = df_quick(s, e);
}

}  // namespace nufft
