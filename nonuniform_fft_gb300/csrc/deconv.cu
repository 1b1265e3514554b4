// Correction steps of the cuFINUFFT paper ("cuFINUFFT: a load-balanced GPU
// library for general-purpose nonuniform FFTs"), row by row:
//   type 1 step 3 (eq. (10)): f_k = p_1(k_1) p_2(k_2) [p_3(k_3)] bhat_{k mod n},
//     truncating the fine-grid spectrum to the central modes k in I_N;
//   type 2 step 1 (eq. (11)): bhat_l = p(k) f_k where l = k mod n for k in I_N,
//     and 0 on every other fine-grid index (pre-correction and zero padding in
//     one pass over the fine grid, so no separate clearing is needed).
// p_i(k) = (2/w) / phihat(alpha_i k), alpha_i = w pi / n_i, is computed once
// per plan on the host and stored per dimension.
#include "nufft_internal.cuh"

namespace nufft {
namespace {

template <typename T> struct C2;
template <> struct C2<float> { using type = float2; };
template <> struct C2<double> { using type = double2; };

struct ModeGeom {
  int N[3];
  int n[3];
  int half[3];  // floor(N_i / 2): mode k has index k + half in f
};

// fine-grid index of output mode index i (0 <= i < N): k = i - half
__device__ __forceinline__ int fine_of_mode(int i, int half, int n) {
  const int k = i - half;
  return k < 0 ? k + n : k;
}

// mode index of fine-grid index l, or -1 when l holds no mode of I_N
__device__ __forceinline__ int mode_of_fine(int l, int N, int half, int n) {
  if (l < N - half) return l + half;       // k = l >= 0
  if (l >= n - half) return l - n + half;  // k = l - n < 0
  return -1;
}

constexpr int kRowThreads = 256;

// Type 1 correction and truncation, one block per chunk of an output row
// (i2, i3): the row's factor p_2 p_3 and its fine-grid row are found once per
// block; along the row the fine-grid reads are two contiguous runs (negative
// modes at the row's end, the others at its start).
template <typename T, int DIM>
__global__ void __launch_bounds__(kRowThreads) deconvolve_kernel(ModeGeom g, const typename C2<T>::type *grid,
                                                                 const T *p1, const T *p2, const T *p3,
                                                                 typename C2<T>::type *f, int bpr,
                                                                 int64_t fstride, int64_t gstride) {
  grid += blockIdx.y * gstride;  // vector blockIdx.y of a batched launch
  f += blockIdx.y * fstride;
  const int row = blockIdx.x / bpr, chunk = blockIdx.x - row * bpr;
  const int i2 = row % g.N[1], i3 = DIM == 3 ? row / g.N[1] : 0;
  const int l2 = fine_of_mode(i2, g.half[1], g.n[1]);
  const int l3 = DIM == 3 ? fine_of_mode(i3, g.half[2], g.n[2]) : 0;
  T s23 = p2[i2];
  if (DIM == 3) s23 *= p3[i3];
  const typename C2<T>::type *grow = grid + (int64_t)g.n[0] * (l2 + (int64_t)g.n[1] * l3);
  typename C2<T>::type *frow = f + (int64_t)g.N[0] * row;
  const int span = (g.N[0] + bpr - 1) / bpr;
  const int a = chunk * span, b = a + span < g.N[0] ? a + span : g.N[0];
  for (int i1 = a + threadIdx.x; i1 < b; i1 += kRowThreads) {
    const typename C2<T>::type v = grow[fine_of_mode(i1, g.half[0], g.n[0])];
    const T s = p1[i1] * s23;
    typename C2<T>::type out;
    out.x = v.x * s;
    out.y = v.y * s;
    frow[i1] = out;
  }
}

// Type 2 correction and zero padding over the whole fine grid, one block per
// chunk of a fine-grid row.  Rows that hold no modes are plain zero stores.
template <typename T, int DIM>
__global__ void __launch_bounds__(kRowThreads) pad_kernel(ModeGeom g, const typename C2<T>::type *f, const T *p1,
                                                          const T *p2, const T *p3, typename C2<T>::type *grid,
                                                          int bpr, int64_t gstride, int64_t fstride) {
  using C = typename C2<T>::type;
  f += blockIdx.y * fstride;  // vector blockIdx.y of a batched launch
  grid += blockIdx.y * gstride;
  const int row = blockIdx.x / bpr, chunk = blockIdx.x - row * bpr;
  const int l2 = row % g.n[1], l3 = DIM == 3 ? row / g.n[1] : 0;
  const int i2 = mode_of_fine(l2, g.N[1], g.half[1], g.n[1]);
  const int i3 = DIM == 3 ? mode_of_fine(l3, g.N[2], g.half[2], g.n[2]) : 0;
  C *grow = grid + (int64_t)g.n[0] * row;
  const int span = (g.n[0] + bpr - 1) / bpr;
  const int a = chunk * span, b = a + span < g.n[0] ? a + span : g.n[0];
  C zero;
  zero.x = zero.y = T(0);
  if (i2 < 0 || i3 < 0) {
    for (int l1 = a + threadIdx.x; l1 < b; l1 += kRowThreads) grow[l1] = zero;
    return;
  }
  T s23 = p2[i2];
  if (DIM == 3) s23 *= p3[i3];
  const C *frow = f + (int64_t)g.N[0] * (i2 + (int64_t)g.N[1] * i3);
  for (int l1 = a + threadIdx.x; l1 < b; l1 += kRowThreads) {
    const int i1 = mode_of_fine(l1, g.N[0], g.half[0], g.n[0]);
    C out = zero;
    if (i1 >= 0) {
      const C v = frow[i1];
      const T s = p1[i1] * s23;
      out.x = v.x * s;
      out.y = v.y * s;
    }
    grow[l1] = out;
  }
}

// Blocks per row: enough chunks of about 8 elements per thread.
inline int chunks_per_row(int64_t len) {
  const int64_t per = 8 * (int64_t)kRowThreads;
  return (int)((len + per - 1) / per > 0 ? (len + per - 1) / per : 1);
}

ModeGeom mode_geom(const nufft_plan_s *p) {
  ModeGeom g;
  for (int d = 0; d < 3; d++) {
    g.N[d] = (int)p->N[d];
    g.n[d] = (int)p->n[d];
    g.half[d] = (int)(p->N[d] / 2);
  }
  return g;
}

template <typename T>
cudaError_t deconv_t(const nufft_plan_s *p, void *f) {
  using C = typename C2<T>::type;
  const int bpr = chunks_per_row(p->N[0]);
  const unsigned blocks = (unsigned)(p->N[1] * p->N[2] * bpr);
  const T *p1 = (const T *)p->pfac[0], *p2 = (const T *)p->pfac[1];
  const T *p3 = (const T *)(p->dim == 3 ? p->pfac[2] : p->pfac[0]);
  if (p->dim <= 2)  // 1D plans carry N2 = n2 = 1 and the factor p2 = 1
    deconvolve_kernel<T, 2><<<dim3(blocks, p->nvec), kRowThreads, 0, p->stream>>>(
        mode_geom(p), (const C *)p->grid, p1, p2, p3, (C *)f, bpr, mode_count(p), grid_cells(p));
  else
    deconvolve_kernel<T, 3><<<dim3(blocks, p->nvec), kRowThreads, 0, p->stream>>>(
        mode_geom(p), (const C *)p->grid, p1, p2, p3, (C *)f, bpr, mode_count(p), grid_cells(p));
  return cudaGetLastError();
}

template <typename T>
cudaError_t pad_t(const nufft_plan_s *p, const void *f) {
  using C = typename C2<T>::type;
  const int bpr = chunks_per_row(p->n[0]);
  const unsigned blocks = (unsigned)(p->n[1] * p->n[2] * bpr);
  const T *p1 = (const T *)p->pfac[0], *p2 = (const T *)p->pfac[1];
  const T *p3 = (const T *)(p->dim == 3 ? p->pfac[2] : p->pfac[0]);
  if (p->dim <= 2)
    pad_kernel<T, 2><<<dim3(blocks, p->nvec), kRowThreads, 0, p->stream>>>(
        mode_geom(p), (const C *)f, p1, p2, p3, (C *)p->grid, bpr, grid_cells(p), mode_count(p));
  else
    pad_kernel<T, 3><<<dim3(blocks, p->nvec), kRowThreads, 0, p->stream>>>(
        mode_geom(p), (const C *)f, p1, p2, p3, (C *)p->grid, bpr, grid_cells(p), mode_count(p));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_deconvolve(const nufft_plan_s *p, void *f) {
  return p->dtype == 0 ? deconv_t<float>(p, f) : deconv_t<double>(p, f);
}

cudaError_t launch_pad(const nufft_plan_s *p, const void *f) {
  return p->dtype == 0 ? pad_t<float>(p, f) : pad_t<double>(p, f);
}

}  // namespace nufft
