// Correction steps of the cuFINUFFT paper ("cuFINUFFT: a load-balanced GPU
// library for general-purpose nonuniform FFTs"), one thread per output value
// as in its Sec. III:
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

template <typename T, int DIM>
__global__ void deconvolve_kernel(ModeGeom g, const typename C2<T>::type *grid, const T *p1,
                                  const T *p2, const T *p3, typename C2<T>::type *f,
                                  int64_t total, int64_t gstride) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  grid += blockIdx.y * gstride;  // vector blockIdx.y of a batched launch
  f += blockIdx.y * total;
  const int i1 = (int)(idx % g.N[0]);
  const int64_t r = idx / g.N[0];
  const int i2 = (int)(r % g.N[1]);
  const int i3 = DIM == 3 ? (int)(r / g.N[1]) : 0;
  const int l1 = fine_of_mode(i1, g.half[0], g.n[0]);
  const int l2 = fine_of_mode(i2, g.half[1], g.n[1]);
  const int l3 = DIM == 3 ? fine_of_mode(i3, g.half[2], g.n[2]) : 0;
  T s = p1[i1] * p2[i2];
  if (DIM == 3) s *= p3[i3];
  const typename C2<T>::type b = grid[l1 + (int64_t)g.n[0] * (l2 + (int64_t)g.n[1] * l3)];
  typename C2<T>::type out;
  out.x = b.x * s;
  out.y = b.y * s;
  f[idx] = out;
}

// mode index of fine-grid index l, or -1 when l holds no mode of I_N
__device__ __forceinline__ int mode_of_fine(int l, int N, int half, int n) {
  if (l < N - half) return l + half;   // k = l >= 0
  if (l >= n - half) return l - n + half;  // k = l - n < 0
  return -1;
}

template <typename T, int DIM>
__global__ void pad_kernel(ModeGeom g, const typename C2<T>::type *f, const T *p1, const T *p2,
                           const T *p3, typename C2<T>::type *grid, int64_t total,
                           int64_t fstride) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  f += blockIdx.y * fstride;  // vector blockIdx.y of a batched launch
  grid += blockIdx.y * total;
  const int l1 = (int)(idx % g.n[0]);
  const int64_t r = idx / g.n[0];
  const int l2 = (int)(r % g.n[1]);
  const int l3 = DIM == 3 ? (int)(r / g.n[1]) : 0;
  const int i1 = mode_of_fine(l1, g.N[0], g.half[0], g.n[0]);
  const int i2 = mode_of_fine(l2, g.N[1], g.half[1], g.n[1]);
  const int i3 = DIM == 3 ? mode_of_fine(l3, g.N[2], g.half[2], g.n[2]) : 0;
  typename C2<T>::type out;
  out.x = T(0);
  out.y = T(0);
  if (i1 >= 0 && i2 >= 0 && i3 >= 0) {
    T s = p1[i1] * p2[i2];
    if (DIM == 3) s *= p3[i3];
    const typename C2<T>::type v = f[i1 + (int64_t)g.N[0] * (i2 + (int64_t)g.N[1] * i3)];
    out.x = v.x * s;
    out.y = v.y * s;
  }
  grid[idx] = out;
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
  const int64_t total = mode_count(p);
  const int threads = 256;
  const unsigned blocks = (unsigned)((total + threads - 1) / threads);
  const T *p1 = (const T *)p->pfac[0], *p2 = (const T *)p->pfac[1];
  const T *p3 = (const T *)(p->dim == 3 ? p->pfac[2] : p->pfac[0]);
  if (p->dim <= 2)  // 1D plans carry N2 = n2 = 1 and the factor p2 = 1
    deconvolve_kernel<T, 2><<<dim3(blocks, p->nvec), threads, 0, p->stream>>>(
        mode_geom(p), (const C *)p->grid, p1, p2, p3, (C *)f, total, grid_cells(p));
  else
    deconvolve_kernel<T, 3><<<dim3(blocks, p->nvec), threads, 0, p->stream>>>(
        mode_geom(p), (const C *)p->grid, p1, p2, p3, (C *)f, total, grid_cells(p));
  return cudaGetLastError();
}

template <typename T>
cudaError_t pad_t(const nufft_plan_s *p, const void *f) {
  using C = typename C2<T>::type;
  const int64_t total = grid_cells(p);
  const int threads = 256;
  const unsigned blocks = (unsigned)((total + threads - 1) / threads);
  const T *p1 = (const T *)p->pfac[0], *p2 = (const T *)p->pfac[1];
  const T *p3 = (const T *)(p->dim == 3 ? p->pfac[2] : p->pfac[0]);
  if (p->dim <= 2)
    pad_kernel<T, 2><<<dim3(blocks, p->nvec), threads, 0, p->stream>>>(
        mode_geom(p), (const C *)f, p1, p2, p3, (C *)p->grid, total, mode_count(p));
  else
    pad_kernel<T, 3><<<dim3(blocks, p->nvec), threads, 0, p->stream>>>(
        mode_geom(p), (const C *)f, p1, p2, p3, (C *)p->grid, total, mode_count(p));
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
