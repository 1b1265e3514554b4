// setpts: bin sort of the nonuniform points and the subproblem table.
//
// Follows Sec. III-A of "cuFINUFFT: a load-balanced GPU library for
// general-purpose nonuniform FFTs" (GM-sort precomputation and SM step 1):
//   1. each point's fine-grid cell, hence its bin (bins of m1 x m2 (x m3)
//      cells, x fastest), and a count per bin;
//   2. an exclusive scan of the counts gives each bin's first sorted slot;
//   3. each point is written to its slot: the permutation t (slot -> user
//      index) and the point's bin-relative grid coordinate;
//   4. each bin's run of points is cut into subproblems of at most M_sub.
//
// The fine-grid coordinate decides integer cells and bins, so it is computed
// in double precision with explicitly rounded operations (no fused
// multiply-add): g = n * frac(x / (2 pi)), node l at l h (eq. (7)).
#include <cmath>

#include "nufft_internal.cuh"

namespace nufft {
namespace {

struct PointsIn {
  const void *x[3];
  int64_t M;
  int dim;
  int is_double;
  double inv_two_pi;
  int n[3];
  int m[3];
  int nb[3];
};

template <typename T>
__device__ __forceinline__ double load_coord(const void *p, int64_t j) {
  return (double)static_cast<const T *>(p)[j];
}

// Fine-grid coordinate in [0, n) of one coordinate; sets *bad for NaN / Inf.
__device__ __forceinline__ double grid_coord(double x, double inv_two_pi, int n, bool *bad) {
  if (!isfinite(x)) {
    *bad = true;
    x = 0.0;
  }
  double t = __dmul_rn(x, inv_two_pi);
  t = __dsub_rn(t, floor(t));
  double g = __dmul_rn(t, (double)n);
  if (g >= (double)n) g = __dsub_rn(g, (double)n);
  return g;
}

template <typename T>
__global__ void bin_count_kernel(PointsIn a, int32_t *counts, int32_t *bin_of, int32_t *rank_of,
                                 int *flag) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= a.M) return;
  bool bad = false;
  int bin = 0, stride = 1;
  for (int d = 0; d < a.dim; d++) {
    double g = grid_coord(load_coord<T>(a.x[d], j), a.inv_two_pi, a.n[d], &bad);
    int cell = (int)floor(g);
    if (cell >= a.n[d]) cell = a.n[d] - 1;  // unreachable; keeps the index in range
    bin += (cell / a.m[d]) * stride;
    stride *= a.nb[d];
  }
  if (bad) atomicOr(flag, 1);
  bin_of[j] = bin;
  rank_of[j] = atomicAdd(&counts[bin], 1);
}

template <typename T>
__global__ void permute_kernel(PointsIn a, const int32_t *starts, const int32_t *bin_of,
                               const int32_t *rank_of, int32_t *perm, T *g0, T *g1, T *g2) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= a.M) return;
  const int32_t pos = starts[bin_of[j]] + rank_of[j];
  perm[pos] = (int32_t)j;
  T *out[3] = {g0, g1, g2};
  bool bad = false;
  for (int d = 0; d < a.dim; d++) {
    double g = grid_coord(load_coord<T>(a.x[d], j), a.inv_two_pi, a.n[d], &bad);
    int cell = (int)floor(g);
    if (cell >= a.n[d]) cell = a.n[d] - 1;
    // bin-relative coordinate in [0, m): exact in double, then rounded to T
    double rel = g - (double)((cell / a.m[d]) * a.m[d]);
    out[d][pos] = (T)rel;
  }
}

__global__ void sub_count_kernel(const int32_t *counts, int64_t nbins, int msub, int32_t *nsub) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nbins) return;
  nsub[b] = (counts[b] + msub - 1) / msub;
}

// One thread per subproblem: find its bin by binary search over the scanned
// subproblem counts, then fill the entry.
__global__ void sub_fill_kernel(const int32_t *counts, const int32_t *starts,
                                const int32_t *sub_starts, int64_t nbins, int64_t nsub, int msub,
                                Subproblem *table) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= nsub) return;
  int64_t lo = 0, hi = nbins - 1;  // last bin b with sub_starts[b] <= s
  while (lo < hi) {
    int64_t mid = (lo + hi + 1) >> 1;
    if (sub_starts[mid] <= s) lo = mid; else hi = mid - 1;
  }
  // skip empty bins that share the same start
  const int64_t b = lo;
  const int32_t k = (int32_t)(s - sub_starts[b]);
  Subproblem e;
  e.bin = (int32_t)b;
  e.start = starts[b] + k * msub;
  const int32_t left = counts[b] - k * msub;
  e.count = left < msub ? left : msub;
  e.pad_ = 0;
  table[s] = e;
}

template <typename Tptr>
cudaError_t grow(Tptr **ptr, int64_t *cap, int64_t need, size_t elem) {
  if (need <= *cap && *ptr) return cudaSuccess;
  if (*ptr) cudaFree(*ptr);
  *ptr = nullptr;
  *cap = 0;
  cudaError_t e = cudaMalloc((void **)ptr, (size_t)(need > 0 ? need : 1) * elem);
  if (e == cudaSuccess) *cap = need;
  return e;
}

}  // namespace

int run_setpts(nufft_plan_s *p, const void *x, const void *y, const void *z) {
  const int64_t M = p->M;
  cudaStream_t s = p->stream;
  const size_t rs = real_size(p);

  // --- storage (grown, never shrunk) --------------------------------------
  if (p->nbins + 1 > p->cap_bins || !p->bin_counts) {
    cudaFree(p->bin_counts);
    cudaFree(p->bin_starts);
    cudaFree(p->sub_counts);
    cudaFree(p->sub_starts);
    cudaFree(p->scan_scratch);
    p->bin_counts = p->bin_starts = p->sub_counts = p->sub_starts = p->scan_scratch = nullptr;
    p->cap_bins = 0;
    const size_t nb = (size_t)(p->nbins + 1) * sizeof(int32_t);
    if (cudaMalloc((void **)&p->bin_counts, nb) != cudaSuccess ||
        cudaMalloc((void **)&p->bin_starts, nb) != cudaSuccess ||
        cudaMalloc((void **)&p->sub_counts, nb) != cudaSuccess ||
        cudaMalloc((void **)&p->sub_starts, nb) != cudaSuccess ||
        cudaMalloc((void **)&p->scan_scratch,
                   (size_t)scan_scratch_len(p->nbins + 1) * sizeof(int32_t)) != cudaSuccess)
      return NUFFT_ERR_ALLOC;
    p->cap_bins = p->nbins + 1;
  }
  if (M > p->cap_pts || !p->perm) {
    cudaFree(p->perm);
    cudaFree(p->bin_of);
    cudaFree(p->rank_of);
    for (int d = 0; d < 3; d++) cudaFree(p->gcoord[d]);
    p->perm = p->bin_of = p->rank_of = nullptr;
    p->gcoord[0] = p->gcoord[1] = p->gcoord[2] = nullptr;
    p->cap_pts = 0;
    const size_t mm = (size_t)(M > 0 ? M : 1);
    if (cudaMalloc((void **)&p->perm, mm * 4) != cudaSuccess ||
        cudaMalloc((void **)&p->bin_of, mm * 4) != cudaSuccess ||
        cudaMalloc((void **)&p->rank_of, mm * 4) != cudaSuccess)
      return NUFFT_ERR_ALLOC;
    for (int d = 0; d < p->dim; d++)
      if (cudaMalloc(&p->gcoord[d], mm * rs) != cudaSuccess) return NUFFT_ERR_ALLOC;
    p->cap_pts = M;
  }
  if (!p->flag && cudaMalloc((void **)&p->flag, sizeof(int)) != cudaSuccess) return NUFFT_ERR_ALLOC;

  // --- 1. bins and counts ------------------------------------------------
  PointsIn a;
  a.x[0] = x;
  a.x[1] = y;
  a.x[2] = p->dim == 3 ? z : x;
  a.M = M;
  a.dim = p->dim;
  a.is_double = p->dtype;
  a.inv_two_pi = 1.0 / (2.0 * 3.14159265358979323846);
  for (int d = 0; d < 3; d++) {
    a.n[d] = (int)p->n[d];
    a.m[d] = p->m[d];
    a.nb[d] = p->nb[d];
  }
  if (cudaMemsetAsync(p->bin_counts, 0, (size_t)(p->nbins + 1) * 4, s) != cudaSuccess ||
      cudaMemsetAsync(p->flag, 0, sizeof(int), s) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  const int threads = 256;
  const unsigned blocks_pts = (unsigned)((M + threads - 1) / threads);
  if (M > 0) {
    if (p->dtype == 0)
      bin_count_kernel<float><<<blocks_pts, threads, 0, s>>>(a, p->bin_counts, p->bin_of, p->rank_of, p->flag);
    else
      bin_count_kernel<double><<<blocks_pts, threads, 0, s>>>(a, p->bin_counts, p->bin_of, p->rank_of, p->flag);
    if (cudaGetLastError() != cudaSuccess) return NUFFT_ERR_CUDA;
  }

  // --- 2. bin starts -------------------------------------------------------
  if (exclusive_scan(p->bin_counts, p->bin_starts, p->nbins, p->scan_scratch, s) != cudaSuccess)
    return NUFFT_ERR_CUDA;

  // --- 3. permutation and sorted coordinates ------------------------------
  if (M > 0) {
    if (p->dtype == 0)
      permute_kernel<float><<<blocks_pts, threads, 0, s>>>(
          a, p->bin_starts, p->bin_of, p->rank_of, p->perm, (float *)p->gcoord[0],
          (float *)p->gcoord[1], (float *)(p->dim == 3 ? p->gcoord[2] : p->gcoord[0]));
    else
      permute_kernel<double><<<blocks_pts, threads, 0, s>>>(
          a, p->bin_starts, p->bin_of, p->rank_of, p->perm, (double *)p->gcoord[0],
          (double *)p->gcoord[1], (double *)(p->dim == 3 ? p->gcoord[2] : p->gcoord[0]));
    if (cudaGetLastError() != cudaSuccess) return NUFFT_ERR_CUDA;
  }

  // --- 4. subproblems ------------------------------------------------------
  const unsigned blocks_bins = (unsigned)((p->nbins + threads - 1) / threads);
  sub_count_kernel<<<blocks_bins, threads, 0, s>>>(p->bin_counts, p->nbins, p->msub, p->sub_counts);
  if (cudaGetLastError() != cudaSuccess) return NUFFT_ERR_CUDA;
  if (exclusive_scan(p->sub_counts, p->sub_starts, p->nbins, p->scan_scratch, s) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  int32_t host_nsub = 0;
  int host_flag = 0;
  if (cudaMemcpyAsync(&host_nsub, p->sub_starts + p->nbins, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(&host_flag, p->flag, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  if (host_flag) return NUFFT_ERR_BAD_POINTS;
  p->nsub = host_nsub;
  if (grow(&p->subprob, &p->cap_sub, p->nsub, sizeof(Subproblem)) != cudaSuccess) return NUFFT_ERR_ALLOC;
  if (p->nsub > 0) {
    sub_fill_kernel<<<(unsigned)((p->nsub + threads - 1) / threads), threads, 0, s>>>(
        p->bin_counts, p->bin_starts, p->sub_starts, p->nbins, p->nsub, p->msub, p->subprob);
    if (cudaGetLastError() != cudaSuccess) return NUFFT_ERR_CUDA;
  }
  return NUFFT_OK;
}

}  // namespace nufft
