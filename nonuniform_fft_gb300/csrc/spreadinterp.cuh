// Spreading (type 1 step 1) and interpolation (type 2 step 3) kernels.
//
// Source: "cuFINUFFT: a load-balanced GPU library for general-purpose
// nonuniform FFTs" (Shih, Wright, Anden, Blaschke, Barnett):
//   - spreading b_l = sum_j c_j psi_per(l h - x_j), eq. (7)-(8), with the ES
//     kernel phi_beta(z) = exp(beta (sqrt(1 - z^2) - 1)), eq. (5);
//   - "SM" (Sec. III-A, Fig. 1): one thread block per subproblem (at most
//     M_sub points of one bin), spreading into a shared-memory copy of the
//     padded bin, p_i = m_i + 2 ceil(w/2) (eq. (13)-(14)), then adding the
//     padded bin back into the fine grid with periodic wrapping (eq. (15));
//   - "GM-sort" (Sec. III-A / III-B): the same sorted traversal without the
//     shared-memory copy, reading / atomically adding the fine grid directly;
//   - interpolation c_j = sum_l b_l psi_per(l h - x_j) (Sec. II-B c) over the
//     sorted points; the SM variant first stages the padded bin of the fine
//     grid in shared memory and then reads only shared memory.
//
// Point data come from setpts: for sorted slot j, perm[j] is the caller's
// index and g_d[j] the coordinate in fine-grid cells relative to the origin
// of the point's bin, in [0, m_d].  Node l (bin-relative) has kernel argument
// z = (l - g) 2 / w; the w nodes taken are l0 .. l0 + w - 1, l0 = ceil(g - w/2),
// i.e. every node with z in [-1, 1).
#pragma once

#include <type_traits>

#include "df64.cuh"
#include "nufft_internal.cuh"

namespace nufft {

template <typename T> struct Cplx;
template <> struct Cplx<float> { using type = float2; };
template <> struct Cplx<double> { using type = double2; };

__device__ __forceinline__ float es_ceil(float v) { return ceilf(v); }
__device__ __forceinline__ double es_ceil(double v) { return ceil(v); }

// ES kernel value phi_beta(z) = exp(beta (sqrt(1 - z^2) - 1)), eq. (5).
// float: hardware approximate square root and base-2 exponential, with
// beta_e = beta * log2(e) folded in; double: the accurate library functions
// with beta_e = beta.  1 - z^2 is formed with one fused multiply-add and
// clamped at 0, so rounding just outside [-1, 1] gives phi = e^-beta.
__device__ __forceinline__ float es_fast(float z, float beta_e) {
  float q = fmaxf(fmaf(-z, z, 1.0f), 0.0f);
  float s, r;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(s) : "f"(q));
  const float arg = fmaf(beta_e, s, -beta_e);
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(arg));
  return r;
}
__device__ __forceinline__ double es_fast(double z, double beta_e) {
  double q = fma(-z, z, 1.0);
  q = q > 0.0 ? q : 0.0;
  return exp(beta_e * (sqrt(q) - 1.0));
}

// beta in the form es_fast takes for precision T.
inline double es_beta_e(double beta, size_t real_bytes) {
  return real_bytes == 4 ? beta * 1.4426950408889634 : beta;
}

// Kernel values of one point in one dimension: k[t] = phi_beta(z_t) for the
// w nodes l0 + t.  Returns l0 (relative to the bin origin).
template <typename T, int W>
__device__ __forceinline__ int es_weights(T g, T beta_e, T (&k)[W]) {
  const T l0 = es_ceil(g - T(0.5) * T(W));
  const T d = l0 - g;
  const T scale = T(2) / T(W);
#pragma unroll
  for (int t = 0; t < W; t++) k[t] = es_fast((d + T(t)) * scale, beta_e);
  return (int)l0;
}

// The same for a given first node l0 (the caller's window origin).
template <typename T, int W>
__device__ __forceinline__ void es_weights_at(T g, int l0, T beta_e, T (&k)[W]) {
  const T d = T(l0) - g;
  const T scale = T(2) / T(W);
#pragma unroll
  for (int t = 0; t < W; t++) k[t] = es_fast((d + T(t)) * scale, beta_e);
}

// The same w kernel values in two-float arithmetic (double-precision plans):
// l0 = ceil(g - w/2) in double, then phi((l0 - g + t) 2/w) by df_es_kernel
// with the table exponential (exp2_64: the 64 values of df_exp2_64, which
// the calling kernel keeps in shared memory).
template <int W>
__device__ __forceinline__ int es_weights_df(double g, DF beta, DF (&k)[W], const DF *exp2_64) {
  const double l0 = ceil(g - 0.5 * W);
  const DF d = df_from(l0 - g);
  const DF scale = df_from(2.0 / W);
#pragma unroll
  for (int t = 0; t < W; t++)
    k[t] = df_es_kernel(df_mul(df_sum(d, DF{(float)t, 0.f}), scale), beta, exp2_64);
  return (int)l0;
}

// Fill a block's shared table of 2^(j/64) (before its first barrier).
__device__ __forceinline__ void fill_exp2_64(DF *tab) {
  for (int j = threadIdx.x; j < 64; j += blockDim.x) tab[j] = df_exp2_64(j);
}

// L2 cache policies.  Points are streamed once per transform (evict first);
// the caller's strengths / results are gathered or scattered through the
// permutation, 8 or 16 bytes per 32-byte sector, so they are kept in L2
// (evict last) until the neighbouring points of the same sector are touched.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ float ld_hint(const float *a, uint64_t pol) {
  float v;
  asm volatile("ld.global.nc.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(a), "l"(pol));
  return v;
}
__device__ __forceinline__ double ld_hint(const double *a, uint64_t pol) {
  double v;
  asm volatile("ld.global.nc.L2::cache_hint.f64 %0, [%1], %2;" : "=d"(v) : "l"(a), "l"(pol));
  return v;
}
__device__ __forceinline__ int32_t ld_hint(const int32_t *a, uint64_t pol) {
  int32_t v;
  asm volatile("ld.global.nc.L2::cache_hint.s32 %0, [%1], %2;" : "=r"(v) : "l"(a), "l"(pol));
  return v;
}
__device__ __forceinline__ float2 ld_hint(const float2 *a, uint64_t pol) {
  float2 v;
  asm volatile("ld.global.nc.L2::cache_hint.v2.f32 {%0, %1}, [%2], %3;"
               : "=f"(v.x), "=f"(v.y) : "l"(a), "l"(pol));
  return v;
}
__device__ __forceinline__ double2 ld_hint(const double2 *a, uint64_t pol) {
  double2 v;
  asm volatile("ld.global.nc.L2::cache_hint.v2.f64 {%0, %1}, [%2], %3;"
               : "=d"(v.x), "=d"(v.y) : "l"(a), "l"(pol));
  return v;
}
__device__ __forceinline__ void st_hint(float2 *a, float2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;"
               :: "l"(a), "f"(v.x), "f"(v.y), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint(double2 *a, double2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.f64 [%0], {%1, %2}, %3;"
               :: "l"(a), "d"(v.x), "d"(v.y), "l"(pol) : "memory");
}

__device__ __forceinline__ void grid_atomic_add(float2 *cell, float re, float im) {
  atomicAdd(cell, make_float2(re, im));
}
__device__ __forceinline__ void grid_atomic_add(double2 *cell, double re, double im) {
  atomicAdd(&cell->x, re);
  atomicAdd(&cell->y, im);
}

// Periodic wrap of a node index that is at most one period out of [0, n)
// (a point's own support: l in [-w, n + w), n >= 2w).
__device__ __forceinline__ int wrap_once(int l, int n) {
  return l < 0 ? l + n : (l >= n ? l - n : l);
}

// Periodic wrap of a padded-tile node, o + s in [-pad, 3n): the last bin of a
// dimension can be narrower than m, so its padded tile may reach past 2n.
__device__ __forceinline__ int wrap_tile(int l, int n) {
  if (l < 0) return l + n;
  while (l >= n) l -= n;
  return l;
}

template <typename T>
struct SIParams {
  using C = typename Cplx<T>::type;
  const Subproblem *sub;
  const int32_t *perm;
  const T *g1, *g2, *g3;
  C *grid;
  const C *c_in;  // type 1 strengths (caller's order)
  C *c_out;       // type 2 results (caller's order)
  T beta;  // in the form es_fast takes (beta * log2(e) for float)
  int n1, n2, n3;
  int m1, m2, m3;
  int nb1, nb2;
  int64_t cstride, gstride;  // per vector: M strengths, one fine grid
};

// Bin coordinates of a bin index (x fastest).
template <int DIM>
__device__ __forceinline__ void bin_coords(int bin, int nb1, int nb2, int &b1, int &b2, int &b3) {
  b1 = bin % nb1;
  const int r = bin / nb1;
  if (DIM == 3) {
    b2 = r % nb2;
    b3 = r / nb2;
  } else {
    b2 = r;
    b3 = 0;
  }
}

// ---------------------------------------------------------------- SM spread
template <typename T, int DIM, int W>
__global__ void spread_sm_kernel(SIParams<T> a) {
  using C = typename Cplx<T>::type;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_in += blockIdx.y * a.cstride;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T *tile = reinterpret_cast<T *>(smem_raw);  // interleaved (re, im)
  constexpr int PAD = (W + 1) / 2;
  const Subproblem sp = a.sub[blockIdx.x];
  int b1, b2, b3;
  bin_coords<DIM>(sp.bin, a.nb1, a.nb2, b1, b2, b3);
  const int p1 = a.m1 + 2 * PAD, p2 = a.m2 + 2 * PAD, p3 = DIM == 3 ? a.m3 + 2 * PAD : 1;
  const int ncell = p1 * p2 * p3;
  for (int i = threadIdx.x; i < 2 * ncell; i += blockDim.x) tile[i] = T(0);
  __syncthreads();

  const int end = sp.start + sp.count;
  for (int j = sp.start + threadIdx.x; j < end; j += blockDim.x) {
    const C cv = a.c_in[a.perm[j]];
    T k1[W], k2[W], k3[W];
    const int s1 = es_weights<T, W>(a.g1[j], a.beta, k1) + PAD;
    const int s2 = es_weights<T, W>(a.g2[j], a.beta, k2) + PAD;
    int s3 = 0;
    if (DIM == 3) s3 = es_weights<T, W>(a.g3[j], a.beta, k3) + PAD;
#pragma unroll 1
    for (int i3 = 0; i3 < (DIM == 3 ? W : 1); i3++) {
      const T v3 = DIM == 3 ? k3[i3] : T(1);
#pragma unroll
      for (int i2 = 0; i2 < W; i2++) {
        const T v = k2[i2] * v3;
        const T vr = cv.x * v, vi = cv.y * v;
        T *row = tile + 2 * (((s3 + i3) * p2 + s2 + i2) * p1 + s1);
#pragma unroll
        for (int i1 = 0; i1 < W; i1++) {
          atomicAdd(row + 2 * i1, vr * k1[i1]);
          atomicAdd(row + 2 * i1 + 1, vi * k1[i1]);
        }
      }
    }
  }
  __syncthreads();

  // add the padded bin back into the fine grid, wrapping periodically (eq. (15))
  const int o1 = b1 * a.m1 - PAD, o2 = b2 * a.m2 - PAD, o3 = DIM == 3 ? b3 * a.m3 - PAD : 0;
  for (int i = threadIdx.x; i < ncell; i += blockDim.x) {
    const T re = tile[2 * i], im = tile[2 * i + 1];
    if (re == T(0) && im == T(0)) continue;
    const int s1 = i % p1;
    const int q = i / p1;
    const int s2 = q % p2;
    const int s3 = q / p2;
    const int l1 = wrap_tile(o1 + s1, a.n1);
    const int l2 = wrap_tile(o2 + s2, a.n2);
    const int l3 = DIM == 3 ? wrap_tile(o3 + s3, a.n3) : 0;
    grid_atomic_add(a.grid + (l1 + (int64_t)a.n1 * (l2 + (int64_t)a.n2 * l3)), re, im);
  }
}

// ---------------------------------------------------------------- GM-sort spread
template <typename T, int DIM, int W>
__global__ void spread_gm_kernel(SIParams<T> a) {
  using C = typename Cplx<T>::type;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_in += blockIdx.y * a.cstride;
  const Subproblem sp = a.sub[blockIdx.x];
  int b1, b2, b3;
  bin_coords<DIM>(sp.bin, a.nb1, a.nb2, b1, b2, b3);
  const int end = sp.start + sp.count;
  for (int j = sp.start + threadIdx.x; j < end; j += blockDim.x) {
    const C cv = a.c_in[a.perm[j]];
    T k1[W], k2[W], k3[W];
    const int l1 = es_weights<T, W>(a.g1[j], a.beta, k1) + b1 * a.m1;
    const int l2 = es_weights<T, W>(a.g2[j], a.beta, k2) + b2 * a.m2;
    int l3 = 0;
    if (DIM == 3) l3 = es_weights<T, W>(a.g3[j], a.beta, k3) + b3 * a.m3;
    int x1[W];
#pragma unroll
    for (int i1 = 0; i1 < W; i1++) x1[i1] = wrap_once(l1 + i1, a.n1);
#pragma unroll 1
    for (int i3 = 0; i3 < (DIM == 3 ? W : 1); i3++) {
      const T v3 = DIM == 3 ? k3[i3] : T(1);
      const int64_t z3 = DIM == 3 ? (int64_t)wrap_once(l3 + i3, a.n3) * a.n2 : 0;
#pragma unroll
      for (int i2 = 0; i2 < W; i2++) {
        const T v = k2[i2] * v3;
        const T vr = cv.x * v, vi = cv.y * v;
        C *row = a.grid + (z3 + wrap_once(l2 + i2, a.n2)) * (int64_t)a.n1;
#pragma unroll
        for (int i1 = 0; i1 < W; i1++) grid_atomic_add(row + x1[i1], vr * k1[i1], vi * k1[i1]);
      }
    }
  }
}

// ---------------------------------------------------------------- SM interp
// Interpolated value of one point from the staged padded bin (Sec. II-B c):
// the w^d tile values around it weighted by the kernel.
template <typename T, int DIM, int W>
__device__ __forceinline__ typename Cplx<T>::type interp_point(const typename Cplx<T>::type *tile,
                                                                int p1, int p2, T gx, T gy, T gz,
                                                                T beta) {
  using C = typename Cplx<T>::type;
  constexpr int PAD = (W + 1) / 2;
  T k1[W], k2[W], k3[W];
  const int s1 = es_weights<T, W>(gx, beta, k1) + PAD;
  const int s2 = es_weights<T, W>(gy, beta, k2) + PAD;
  int s3 = 0;
  if (DIM == 3) s3 = es_weights<T, W>(gz, beta, k3) + PAD;
  T ar = T(0), ai = T(0);
#pragma unroll 1
  for (int i3 = 0; i3 < (DIM == 3 ? W : 1); i3++) {
    T sr3 = T(0), si3 = T(0);
#pragma unroll
    for (int i2 = 0; i2 < W; i2++) {
      const C *row = tile + ((s3 + i3) * p2 + s2 + i2) * p1 + s1;
      T sr = T(0), si = T(0);
#pragma unroll
      for (int i1 = 0; i1 < W; i1++) {
        const C b = row[i1];
        sr += b.x * k1[i1];
        si += b.y * k1[i1];
      }
      sr3 += sr * k2[i2];
      si3 += si * k2[i2];
    }
    const T v3 = DIM == 3 ? k3[i3] : T(1);
    ar += sr3 * v3;
    ai += si3 * v3;
  }
  C out;
  out.x = ar;
  out.y = ai;
  return out;
}

template <typename T, int DIM, int W>
__global__ void interp_sm_kernel(SIParams<T> a) {
  using C = typename Cplx<T>::type;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_out += blockIdx.y * a.cstride;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  C *tile = reinterpret_cast<C *>(smem_raw);
  constexpr int PAD = (W + 1) / 2;
  const Subproblem sp = a.sub[blockIdx.x];
  int b1, b2, b3;
  bin_coords<DIM>(sp.bin, a.nb1, a.nb2, b1, b2, b3);
  const int p1 = a.m1 + 2 * PAD, p2 = a.m2 + 2 * PAD, p3 = DIM == 3 ? a.m3 + 2 * PAD : 1;
  const int o1 = b1 * a.m1 - PAD, o2 = b2 * a.m2 - PAD, o3 = DIM == 3 ? b3 * a.m3 - PAD : 0;
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int end = sp.start + sp.count;
  const int stride = 2 * blockDim.x;

  // the first two points' coordinates and destinations are requested before
  // the tile, so their latency overlaps the staging
  T nx[2] = {T(0), T(0)}, ny[2] = {T(0), T(0)}, nz[2] = {T(0), T(0)};
  int nd[2] = {0, 0};
  int j = sp.start + threadIdx.x;
#pragma unroll
  for (int u = 0; u < 2; u++) {
    const int jj = j + u * (int)blockDim.x;
    if (jj < end) {
      nx[u] = ld_hint(a.g1 + jj, pol_stream);
      ny[u] = ld_hint(a.g2 + jj, pol_stream);
      if (DIM == 3) nz[u] = ld_hint(a.g3 + jj, pol_stream);
      nd[u] = ld_hint(a.perm + jj, pol_stream);
    }
  }

  // stage the padded bin of the fine grid (periodic wrap) in shared memory:
  // one warp per tile row, lanes along the row (no division per cell), four
  // rows' loads in flight per lane before their stores
  {
    const int rows = p2 * p3, nw = blockDim.x >> 5, lane = threadIdx.x & 31;
    for (int r0 = threadIdx.x >> 5; r0 < rows; r0 += 4 * nw) {
      for (int c = lane; c < p1; c += 32) {
        const int l1 = wrap_tile(o1 + c, a.n1);
        C v[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
          const int r = r0 + u * nw;
          if (r < rows) {
            const int s2 = DIM == 3 ? r % p2 : r, s3 = DIM == 3 ? r / p2 : 0;
            const int l2 = wrap_tile(o2 + s2, a.n2);
            const int l3 = DIM == 3 ? wrap_tile(o3 + s3, a.n3) : 0;
            v[u] = a.grid[l1 + (int64_t)a.n1 * (l2 + (int64_t)a.n2 * l3)];
          }
        }
#pragma unroll
        for (int u = 0; u < 4; u++)
          if (r0 + u * nw < rows) tile[(r0 + u * nw) * p1 + c] = v[u];
      }
    }
  }
  __syncthreads();

  // two points per thread and iteration, the next two prefetched
  for (; j < end; j += stride) {
    T gx[2], gy[2], gz[2];
    int dst[2];
#pragma unroll
    for (int u = 0; u < 2; u++) {
      gx[u] = nx[u];
      gy[u] = ny[u];
      gz[u] = nz[u];
      dst[u] = nd[u];
    }
#pragma unroll
    for (int u = 0; u < 2; u++) {
      const int jn = j + stride + u * (int)blockDim.x;
      if (jn < end) {
        nx[u] = ld_hint(a.g1 + jn, pol_stream);
        ny[u] = ld_hint(a.g2 + jn, pol_stream);
        if (DIM == 3) nz[u] = ld_hint(a.g3 + jn, pol_stream);
        nd[u] = ld_hint(a.perm + jn, pol_stream);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; u++) {
      if (j + u * (int)blockDim.x < end) {
        const C out = interp_point<T, DIM, W>(tile, p1, p2, gx[u], gy[u], gz[u], a.beta);
        st_hint(a.c_out + dst[u], out, pol_keep);
      }
    }
  }
}

// Single precision in 3D: the staged tile and thread-per-point sums of
// interp_sm_kernel, with the subproblem's points taken in a bank-spread
// order.  A point's w^3 tile reads all fall on bank pair (window origin +
// common offset) mod 16, so 16 lanes of a half warp whose window origins are
// distinct mod 16 read without bank conflicts.  The block buckets its points
// by origin mod 16 (a counting sort in shared memory) and walks the
// bucket-sorted list with a stride close to n / 16 and coprime with n, so
// consecutive lanes take points from consecutive buckets.  In cell order the
// windows of neighbouring points start on different rows and planes, and the
// loads average 4.5 wavefronts per warp instruction instead of 2.
template <int W>
__global__ void interp_sm3d_bank_kernel(SIParams<float> a) {
  using C = float2;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_out += blockIdx.y * a.cstride;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int PAD = (W + 1) / 2;
  const Subproblem sp = a.sub[blockIdx.x];
  int b1, b2, b3;
  bin_coords<3>(sp.bin, a.nb1, a.nb2, b1, b2, b3);
  const int p1 = a.m1 + 2 * PAD, p2 = a.m2 + 2 * PAD, p3 = a.m3 + 2 * PAD;
  const int o1 = b1 * a.m1 - PAD, o2 = b2 * a.m2 - PAD, o3 = b3 * a.m3 - PAD;
  const int cells = p1 * p2 * p3;
  C *tile = reinterpret_cast<C *>(smem_raw);
  int *order = reinterpret_cast<int *>(tile + cells);  // sp.count entries
  __shared__ int cnt[16], cur[16], step_s;
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int n = sp.count;
  if (threadIdx.x < 16) cnt[threadIdx.x] = 0;
  for (int base = threadIdx.x; base < cells; base += 4 * blockDim.x) {
    C v[4];
    int at[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int t = base + u * (int)blockDim.x;
      at[u] = t;
      if (t < cells) {
        const int s1 = t % p1, rr = t / p1;
        const int s2 = rr % p2, s3 = rr / p2;
        v[u] = a.grid[wrap_tile(o1 + s1, a.n1) +
                      (int64_t)a.n1 * (wrap_tile(o2 + s2, a.n2) + (int64_t)a.n2 * wrap_tile(o3 + s3, a.n3))];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; u++)
      if (at[u] < cells) tile[at[u]] = v[u];
  }
  __syncthreads();
  // window origin of a point in the tile, and its bank pair
  auto origin = [&](int k) {
    const int j = sp.start + k;
    const int s1 = (int)es_ceil(a.g1[j] - 0.5f * W) + PAD;
    const int s2 = (int)es_ceil(a.g2[j] - 0.5f * W) + PAD;
    const int s3 = (int)es_ceil(a.g3[j] - 0.5f * W) + PAD;
    return (s3 * p2 + s2) * p1 + s1;
  };
  for (int k = threadIdx.x; k < n; k += blockDim.x) atomicAdd(&cnt[origin(k) & 15], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < 16; b++) {
      cur[b] = acc;
      acc += cnt[b];
    }
    int st = n / 16 > 0 ? n / 16 : 1;
    auto gcd = [](int x, int y) {
      while (y) {
        const int t = x % y;
        x = y;
        y = t;
      }
      return x;
    };
    while (gcd(st, n) != 1) st++;
    step_s = st;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < n; k += blockDim.x) order[atomicAdd(&cur[origin(k) & 15], 1)] = k;
  __syncthreads();

  const int step = step_s;
  // slot s takes order[(s step) mod n], updated incrementally
  int idx = n > 0 ? (int)(((int64_t)threadIdx.x * step) % n) : 0;
  const int inc = n > 0 ? (int)(((int64_t)blockDim.x * step) % n) : 0;
  for (int slot = threadIdx.x; slot < n; slot += blockDim.x) {
    const int k = order[idx];
    idx += inc;
    if (idx >= n) idx -= n;
    const int j = sp.start + k;
    const C out = interp_point<float, 3, W>(tile, p1, p2, ld_hint(a.g1 + j, pol_stream),
                                            ld_hint(a.g2 + j, pol_stream), ld_hint(a.g3 + j, pol_stream),
                                            a.beta);
    st_hint(a.c_out + ld_hint(a.perm + j, pol_stream), out, pol_keep);
  }
}

// Double precision in 3D: the same staged tile and thread-per-point sums, with
// the w^3 multiply-accumulates in two-float arithmetic (df64.cuh).  The tile
// is converted to two-floats once when it is staged; the kernel values are
// evaluated in double and split once per point.
struct DFC2 {  // complex two-float, 16 bytes
  DF re, im;
};

template <int W>
__global__ void __launch_bounds__(640, 1) interp_sm3d_df_kernel(SIParams<double> a) {
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_out += blockIdx.y * a.cstride;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  DFC2 *tile = reinterpret_cast<DFC2 *>(smem_raw);
  __shared__ DF s_exp2[64];
  fill_exp2_64(s_exp2);
  constexpr int PAD = (W + 1) / 2;
  const Subproblem sp = a.sub[blockIdx.x];
  int b1, b2, b3;
  bin_coords<3>(sp.bin, a.nb1, a.nb2, b1, b2, b3);
  const int p1 = a.m1 + 2 * PAD, p2 = a.m2 + 2 * PAD, p3 = a.m3 + 2 * PAD;
  const int o1 = b1 * a.m1 - PAD, o2 = b2 * a.m2 - PAD, o3 = b3 * a.m3 - PAD;
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  {
    const int cells = p1 * p2 * p3;
    for (int base = threadIdx.x; base < cells; base += 4 * blockDim.x) {
      double2 v[4];
      int at[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int t = base + u * (int)blockDim.x;
        at[u] = t;
        if (t < cells) {
          const int s1 = t % p1, r = t / p1;
          const int s2 = r % p2, s3 = r / p2;
          const int l1 = wrap_tile(o1 + s1, a.n1);
          const int l2 = wrap_tile(o2 + s2, a.n2);
          const int l3 = wrap_tile(o3 + s3, a.n3);
          v[u] = a.grid[l1 + (int64_t)a.n1 * (l2 + (int64_t)a.n2 * l3)];
        }
      }
#pragma unroll
      for (int u = 0; u < 4; u++)
        if (at[u] < cells) {
          DFC2 d;
          d.re = df_from(v[u].x);
          d.im = df_from(v[u].y);
          tile[at[u]] = d;
        }
    }
  }
  __syncthreads();
  const int end = sp.start + sp.count;
  for (int j = sp.start + threadIdx.x; j < end; j += blockDim.x) {
    DF kx[W], ky[W], kz[W];
    const DF beta = df_from(a.beta);
    const int s1 = es_weights_df<W>(ld_hint(a.g1 + j, pol_stream), beta, kx, s_exp2) + PAD;
    const int s2 = es_weights_df<W>(ld_hint(a.g2 + j, pol_stream), beta, ky, s_exp2) + PAD;
    const int s3 = es_weights_df<W>(ld_hint(a.g3 + j, pol_stream), beta, kz, s_exp2) + PAD;
    const int dst = ld_hint(a.perm + j, pol_stream);
    DF ar{0.f, 0.f}, ai{0.f, 0.f};
#pragma unroll 1
    for (int i3 = 0; i3 < W; i3++) {
      DF r3{0.f, 0.f}, i3s{0.f, 0.f};
#pragma unroll
      for (int i2 = 0; i2 < W; i2++) {
        const DFC2 *row = tile + ((s3 + i3) * p2 + s2 + i2) * p1 + s1;
        // two independent chains per component (even and odd i1), each at
        // most 8 terms, renormalised when the two are added
        DF sr0{0.f, 0.f}, si0{0.f, 0.f}, sr1{0.f, 0.f}, si1{0.f, 0.f};
#pragma unroll
        for (int i1 = 0; i1 < W; i1 += 2) {
          const DFC2 b = row[i1];
          df_fma_lazy(sr0, b.re, kx[i1]);
          df_fma_lazy(si0, b.im, kx[i1]);
          if (i1 + 1 < W) {
            const DFC2 c = row[i1 + 1];
            df_fma_lazy(sr1, c.re, kx[i1 + 1]);
            df_fma_lazy(si1, c.im, kx[i1 + 1]);
          }
        }
        df_fma(r3, df_sum(sr0, sr1), ky[i2]);
        df_fma(i3s, df_sum(si0, si1), ky[i2]);
      }
      df_fma(ar, r3, kz[i3]);
      df_fma(ai, i3s, kz[i3]);
    }
    double2 out;
    out.x = df_to(ar);
    out.y = df_to(ai);
    st_hint(a.c_out + dst, out, pol_keep);
  }
}

template <typename T, int DIM, int W>
__global__ void interp_gm_kernel(SIParams<T> a) {
  using C = typename Cplx<T>::type;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_out += blockIdx.y * a.cstride;
  const Subproblem sp = a.sub[blockIdx.x];
  int b1, b2, b3;
  bin_coords<DIM>(sp.bin, a.nb1, a.nb2, b1, b2, b3);
  const int end = sp.start + sp.count;
  for (int j = sp.start + threadIdx.x; j < end; j += blockDim.x) {
    T k1[W], k2[W], k3[W];
    const int l1 = es_weights<T, W>(a.g1[j], a.beta, k1) + b1 * a.m1;
    const int l2 = es_weights<T, W>(a.g2[j], a.beta, k2) + b2 * a.m2;
    int l3 = 0;
    if (DIM == 3) l3 = es_weights<T, W>(a.g3[j], a.beta, k3) + b3 * a.m3;
    int x1[W];
#pragma unroll
    for (int i1 = 0; i1 < W; i1++) x1[i1] = wrap_once(l1 + i1, a.n1);
    T ar = T(0), ai = T(0);
#pragma unroll 1
    for (int i3 = 0; i3 < (DIM == 3 ? W : 1); i3++) {
      const int64_t z3 = DIM == 3 ? (int64_t)wrap_once(l3 + i3, a.n3) * a.n2 : 0;
      T sr3 = T(0), si3 = T(0);
#pragma unroll
      for (int i2 = 0; i2 < W; i2++) {
        const C *row = a.grid + (z3 + wrap_once(l2 + i2, a.n2)) * (int64_t)a.n1;
        T sr = T(0), si = T(0);
#pragma unroll
        for (int i1 = 0; i1 < W; i1++) {
          const C b = __ldg(row + x1[i1]);
          sr += b.x * k1[i1];
          si += b.y * k1[i1];
        }
        sr3 += sr * k2[i2];
        si3 += si * k2[i2];
      }
      const T v3 = DIM == 3 ? k3[i3] : T(1);
      ar += sr3 * v3;
      ai += si3 * v3;
    }
    C out;
    out.x = ar;
    out.y = ai;
    a.c_out[a.perm[j]] = out;
  }
}

// ---------------------------------------------------------------- GM (unsorted)
// [cuFINUFFT] Sec. III-A "GM": one thread per point in the caller's order,
// every kernel-weighted value added straight into the fine grid with a
// global atomic; Sec. III-B "GM" interpolation reads the fine grid directly.
// No bin sort: setpts only stores each point's fine-grid cell (packed
// l1 + n1 (l2 + n2 l3), in the `perm` slot of the parameters) and its
// fractional position inside the cell (in g1..g3), in the caller's order.
template <typename T, int DIM>
__device__ __forceinline__ void unpack_cell(int packed, int n1, int n2, int &l1, int &l2, int &l3) {
  l1 = packed % n1;
  const int r = packed / n1;
  if (DIM == 3) {
    l2 = r % n2;
    l3 = r / n2;
  } else {
    l2 = r;
    l3 = 0;
  }
}

template <typename T, int DIM, int W>
__global__ void spread_gmu_kernel(SIParams<T> a, int64_t M) {
  using C = typename Cplx<T>::type;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_in += blockIdx.y * a.cstride;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= M) return;
  int c1, c2, c3;
  unpack_cell<T, DIM>(a.perm[i], a.n1, a.n2, c1, c2, c3);
  const C cv = a.c_in[i];
  T k1[W], k2[W], k3[W];
  const int l1 = es_weights<T, W>(a.g1[i], a.beta, k1) + c1;
  const int l2 = es_weights<T, W>(a.g2[i], a.beta, k2) + c2;
  int l3 = 0;
  if (DIM == 3) l3 = es_weights<T, W>(a.g3[i], a.beta, k3) + c3;
  int x1[W];
#pragma unroll
  for (int i1 = 0; i1 < W; i1++) x1[i1] = wrap_once(l1 + i1, a.n1);
#pragma unroll 1
  for (int i3 = 0; i3 < (DIM == 3 ? W : 1); i3++) {
    const T v3 = DIM == 3 ? k3[i3] : T(1);
    const int64_t z3 = DIM == 3 ? (int64_t)wrap_once(l3 + i3, a.n3) * a.n2 : 0;
#pragma unroll
    for (int i2 = 0; i2 < W; i2++) {
      const T v = k2[i2] * v3;
      const T vr = cv.x * v, vi = cv.y * v;
      C *row = a.grid + (z3 + wrap_once(l2 + i2, a.n2)) * (int64_t)a.n1;
#pragma unroll
      for (int i1 = 0; i1 < W; i1++) grid_atomic_add(row + x1[i1], vr * k1[i1], vi * k1[i1]);
    }
  }
}

template <typename T, int DIM, int W>
__global__ void interp_gmu_kernel(SIParams<T> a, int64_t M) {
  using C = typename Cplx<T>::type;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_out += blockIdx.y * a.cstride;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= M) return;
  int c1, c2, c3;
  unpack_cell<T, DIM>(a.perm[i], a.n1, a.n2, c1, c2, c3);
  T k1[W], k2[W], k3[W];
  const int l1 = es_weights<T, W>(a.g1[i], a.beta, k1) + c1;
  const int l2 = es_weights<T, W>(a.g2[i], a.beta, k2) + c2;
  int l3 = 0;
  if (DIM == 3) l3 = es_weights<T, W>(a.g3[i], a.beta, k3) + c3;
  int x1[W];
#pragma unroll
  for (int i1 = 0; i1 < W; i1++) x1[i1] = wrap_once(l1 + i1, a.n1);
  T ar = T(0), ai = T(0);
#pragma unroll 1
  for (int i3 = 0; i3 < (DIM == 3 ? W : 1); i3++) {
    const int64_t z3 = DIM == 3 ? (int64_t)wrap_once(l3 + i3, a.n3) * a.n2 : 0;
    T sr3 = T(0), si3 = T(0);
#pragma unroll
    for (int i2 = 0; i2 < W; i2++) {
      const C *row = a.grid + (z3 + wrap_once(l2 + i2, a.n2)) * (int64_t)a.n1;
      T sr = T(0), si = T(0);
#pragma unroll
      for (int i1 = 0; i1 < W; i1++) {
        const C b = __ldg(row + x1[i1]);
        sr += b.x * k1[i1];
        si += b.y * k1[i1];
      }
      sr3 += sr * k2[i2];
      si3 += si * k2[i2];
    }
    const T v3 = DIM == 3 ? k3[i3] : T(1);
    ar += sr3 * v3;
    ai += si3 * v3;
  }
  C out;
  out.x = ar;
  out.y = ai;
  a.c_out[i] = out;
}

// ---------------------------------------------------------------- launchers

template <typename T>
SIParams<T> make_params(const nufft_plan_s *p) {
  SIParams<T> a{};
  a.sub = p->subprob;
  a.perm = p->perm;
  a.g1 = static_cast<const T *>(p->gcoord[0]);
  a.g2 = static_cast<const T *>(p->gcoord[1]);
  a.g3 = static_cast<const T *>(p->dim == 3 ? p->gcoord[2] : p->gcoord[0]);
  a.grid = static_cast<typename Cplx<T>::type *>(p->grid);
  a.c_in = nullptr;
  a.c_out = nullptr;
  a.beta = (T)es_beta_e(p->beta, sizeof(T));
  a.n1 = (int)p->n[0];
  a.n2 = (int)p->n[1];
  a.n3 = (int)p->n[2];
  a.m1 = p->m[0];
  a.m2 = p->m[1];
  a.m3 = p->m[2];
  a.nb1 = p->nb[0];
  a.nb2 = p->nb[1];
  a.cstride = p->M;
  a.gstride = grid_cells(p);
  return a;
}

inline size_t tile_cells(const nufft_plan_s *p) {
  const int pad = (p->w + 1) / 2;
  size_t cells = 1;
  for (int d = 0; d < p->dim; d++) cells *= (size_t)(p->m[d] + 2 * pad);
  return cells;
}

// Threads per block for a kernel: the requested count, lowered (in whole
// warps) to what the kernel's register use allows.
template <typename Kern>
int block_threads(Kern kern, int requested) {
  cudaFuncAttributes at;
  if (cudaFuncGetAttributes(&at, kern) != cudaSuccess) return requested;
  const int cap = at.maxThreadsPerBlock / 32 * 32;
  return requested < cap ? requested : cap;
}

// Kernels that need more than the default 48 KB of dynamic shared memory must
// opt in before launch.
template <typename Kern>
cudaError_t allow_smem(Kern kern, size_t smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <int DIM, typename T, int W>
cudaError_t spread_w(const nufft_plan_s *p, const void *c) {
  SIParams<T> a = make_params<T>(p);
  a.c_in = static_cast<const typename Cplx<T>::type *>(c);
  const unsigned blocks = (unsigned)p->nsub;
  if (p->method == NUFFT_METHOD_GM) {
    a.perm = p->bin_of;  // packed cells, caller's order
    const int th = block_threads(spread_gmu_kernel<T, DIM, W>, p->threads);
    spread_gmu_kernel<T, DIM, W><<<dim3((unsigned)((p->M + th - 1) / th), p->nvec), th, 0,
                                   p->stream>>>(a, p->M);
    return cudaGetLastError();
  }
  if (p->method == NUFFT_METHOD_GM_SORT) {
    spread_gm_kernel<T, DIM, W><<<dim3(blocks, p->nvec), block_threads(spread_gm_kernel<T, DIM, W>, p->threads),
                                  0, p->stream>>>(a);
    return cudaGetLastError();
  }
  const size_t smem = tile_cells(p) * 2 * sizeof(T);
  cudaError_t e = allow_smem(spread_sm_kernel<T, DIM, W>, smem);
  if (e != cudaSuccess) return e;
  spread_sm_kernel<T, DIM, W><<<dim3(blocks, p->nvec), block_threads(spread_sm_kernel<T, DIM, W>, p->threads),
                                smem, p->stream>>>(a);
  return cudaGetLastError();
}

template <int DIM, typename T, int W>
cudaError_t interp_w(const nufft_plan_s *p, void *c) {
  SIParams<T> a = make_params<T>(p);
  a.c_out = static_cast<typename Cplx<T>::type *>(c);
  const unsigned blocks = (unsigned)p->nsub;
  if (p->method == NUFFT_METHOD_GM) {
    a.perm = p->bin_of;  // packed cells, caller's order
    const int th = block_threads(interp_gmu_kernel<T, DIM, W>, p->threads);
    interp_gmu_kernel<T, DIM, W><<<dim3((unsigned)((p->M + th - 1) / th), p->nvec), th, 0,
                                   p->stream>>>(a, p->M);
    return cudaGetLastError();
  }
  if (p->method == NUFFT_METHOD_GM_SORT) {
    interp_gm_kernel<T, DIM, W><<<dim3(blocks, p->nvec), block_threads(interp_gm_kernel<T, DIM, W>, p->threads),
                                  0, p->stream>>>(a);
    return cudaGetLastError();
  }
  const size_t smem = tile_cells(p) * 2 * sizeof(T);
  if constexpr (DIM == 3 && std::is_same<T, float>::value) {
    const size_t smem_bk = smem + (size_t)p->msub * sizeof(int);
    cudaError_t e = allow_smem(interp_sm3d_bank_kernel<W>, smem_bk);
    if (e != cudaSuccess) return e;
    interp_sm3d_bank_kernel<W><<<dim3(blocks, p->nvec), block_threads(interp_sm3d_bank_kernel<W>, p->threads),
                                 smem_bk, p->stream>>>(a);
    return cudaGetLastError();
  }
  if constexpr (DIM == 3 && std::is_same<T, double>::value) {
    cudaError_t e = allow_smem(interp_sm3d_df_kernel<W>, smem);
    if (e != cudaSuccess) return e;
    interp_sm3d_df_kernel<W><<<dim3(blocks, p->nvec), block_threads(interp_sm3d_df_kernel<W>, p->threads),
                               smem, p->stream>>>(a);
  } else {
    cudaError_t e = allow_smem(interp_sm_kernel<T, DIM, W>, smem);
    if (e != cudaSuccess) return e;
    interp_sm_kernel<T, DIM, W><<<dim3(blocks, p->nvec), block_threads(interp_sm_kernel<T, DIM, W>, p->threads),
                                  smem, p->stream>>>(a);
  }
  return cudaGetLastError();
}

// Dispatch on the kernel width (compile-time in the kernels).
template <int DIM, typename T>
cudaError_t launch_spread_t(const nufft_plan_s *p, const void *c) {
  switch (p->w) {
    case 2: return spread_w<DIM, T, 2>(p, c);
    case 3: return spread_w<DIM, T, 3>(p, c);
    case 4: return spread_w<DIM, T, 4>(p, c);
    case 5: return spread_w<DIM, T, 5>(p, c);
    case 6: return spread_w<DIM, T, 6>(p, c);
    case 7: return spread_w<DIM, T, 7>(p, c);
    case 8: return spread_w<DIM, T, 8>(p, c);
    case 9: return spread_w<DIM, T, 9>(p, c);
    case 10: return spread_w<DIM, T, 10>(p, c);
    case 11: return spread_w<DIM, T, 11>(p, c);
    case 12: return spread_w<DIM, T, 12>(p, c);
    case 13: return spread_w<DIM, T, 13>(p, c);
    case 14: return spread_w<DIM, T, 14>(p, c);
    case 15: return spread_w<DIM, T, 15>(p, c);
    case 16: return spread_w<DIM, T, 16>(p, c);
    default: return cudaErrorInvalidValue;
  }
}

template <int DIM, typename T>
cudaError_t launch_interp_t(const nufft_plan_s *p, void *c) {
  switch (p->w) {
    case 2: return interp_w<DIM, T, 2>(p, c);
    case 3: return interp_w<DIM, T, 3>(p, c);
    case 4: return interp_w<DIM, T, 4>(p, c);
    case 5: return interp_w<DIM, T, 5>(p, c);
    case 6: return interp_w<DIM, T, 6>(p, c);
    case 7: return interp_w<DIM, T, 7>(p, c);
    case 8: return interp_w<DIM, T, 8>(p, c);
    case 9: return interp_w<DIM, T, 9>(p, c);
    case 10: return interp_w<DIM, T, 10>(p, c);
    case 11: return interp_w<DIM, T, 11>(p, c);
    case 12: return interp_w<DIM, T, 12>(p, c);
    case 13: return interp_w<DIM, T, 13>(p, c);
    case 14: return interp_w<DIM, T, 14>(p, c);
    case 15: return interp_w<DIM, T, 15>(p, c);
    case 16: return interp_w<DIM, T, 16>(p, c);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nufft
