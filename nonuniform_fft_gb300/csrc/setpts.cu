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
#include <mutex>
#include <type_traits>

#include "nufft_internal.cuh"

namespace nufft {
namespace {

struct PointsIn {
  const void *x[3];
  int64_t M;
  int dim;
  int is_double;
  double inv_two_pi;
  float turn3[3];  // inv_two_pi split exactly into three floats (fold_fast)
  int fast;        // 1: turn3 is exact, so fold_fast may be used
  int origin;      // 1: bin by window origin (origin_node), 0: by cell
  float oc;        // origin_node offset: 1/2 for odd w, 0 for even w
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

// Sum of two floats as an unevaluated pair hi + lo, exactly (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float *hi, float *lo) {
  const float s = a + b;
  const float bv = s - a;
  *lo = (a - (s - bv)) + (b - bv);
  *hi = s;
}

// The fold of a single-precision coordinate without FP64 arithmetic: g ~
// n frac(x inv_two_pi) as gh + gl, from exact float products of x with the
// three-float split of the double inv_two_pi (x c0 and x c1 each as a
// product and its fused-multiply-add error; x c2 rounded; the fraction of
// the leading product as a TwoSum pair).  The result is within
// n (2.5e-14 |x c| + 9e-15) of the double fold grid_coord computes
// (its own two roundings included), so when gh + gl lies farther than twice
// that from every integer, floor(g) -- the cell -- is the same as the double
// fold's.  Returns false, for the caller to take the double fold, when x is
// not finite, |x| > 1024, n >= 2^24, or g is that close to a cell boundary
// (about 1e-8 of the coordinates at n = 2048).  Otherwise sets the cell and
// gh + gl (no part of the integer result depends on gl beyond the check).
__device__ __forceinline__ bool fold_fast_hl(float x, const float (&c)[3], int n, float *gh, float *gl,
                                             float *delta) {
  if (!(fabsf(x) <= 1024.0f) || n >= (1 << 24)) return false;
  const float p0 = x * c[0], e0 = fmaf(x, c[0], -p0);
  const float p1 = x * c[1], e1 = fmaf(x, c[1], -p1);
  const float p2 = x * c[2];
  float f, fl;
  two_sum(p0, -floorf(p0), &f, &fl);  // p0 - floor(p0) = f + fl exactly (f in [0, 1])
  const float tail = ((e0 + p1) + (e1 + p2)) + fl;
  float s, sl;
  two_sum(f, tail, &s, &sl);  // frac(x c) up to an integer
  if (s < 0.0f) {
    float t, tl;
    two_sum(s, 1.0f, &t, &tl);
    s = t;
    sl += tl;
  } else if (s >= 1.0f) {
    float t, tl;
    two_sum(s, -1.0f, &t, &tl);
    s = t;
    sl += tl;
  }
  const float nf = (float)n;
  const float h = s * nf;
  *gl = fmaf(s, nf, -h) + sl * nf;
  *gh = h;
  *delta = nf * (fabsf(p0) + 1.0f) * 5.6843419e-14f;  // n (|x c| + 1) 2^-44
  return true;
}

// The cell floor(g) of g = gh + gl (fold_fast_hl), when g is farther than
// delta from every integer.
__device__ __forceinline__ bool cell_from_hl(float h, float l, float delta, int n, int *cell) {
  const float r = rintf(h);
  const float d = (h - r) + l;  // h - r is exact
  if (fabsf(d) <= delta) return false;
  const int k = (int)r - (d < 0.0f ? 1 : 0);
  if (k < 0 || k >= n) return false;
  *cell = k;
  return true;
}

// The node ceil(g - oc), in [0, n], of g = gh + gl (fold_fast_hl), when g -
// oc is farther than delta from every integer (oc = 1/2 or 0; h - 1/2 is
// exact below 2^22).
__device__ __forceinline__ bool node_from_hl(float h, float l, float delta, float oc, int n, int *node) {
  if (oc != 0.0f && n > (1 << 22)) return false;
  const float h2 = h - oc;
  const float r = rintf(h2);
  const float d = (h2 - r) + l;
  if (fabsf(d) <= delta) return false;
  const int k = (int)r + (d > 0.0f ? 1 : 0);
  if (k < 0 || k > n) return false;
  *node = k;
  return true;
}

__device__ __forceinline__ bool fold_fast(float x, const float (&c)[3], int n, int *cell, float *gh,
                                          float *gl) {
  float delta;
  return fold_fast_hl(x, c, n, gh, gl, &delta) && cell_from_hl(*gh, *gl, delta, n, cell);
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

__device__ __forceinline__ float below(float v) { return nextafterf(v, 0.0f); }
__device__ __forceinline__ double below(double v) { return ::nextafter(v, 0.0); }

// Cell-level key of a point: its bin, then its cell inside the bin (x fastest).
// Sorting by this key orders the points bin by bin (as Sec. III-A) and, inside
// each bin, cell by cell, so a bin's points of one fine-grid row (and one x
// range of that row) form a contiguous run.
// The fold to the fine grid is done once, here: the point's bin-relative
// coordinate, rounded to T but never up to the next cell (floor stays the
// point's cell), is written in the caller's order to rel_d and later gathered
// into sorted order.
// A point's bin-relative coordinates as one record of setpts' scratch: DIM
// values, padded to 4 in 3D, so that gathering a point's record through the
// permutation touches one 32-byte sector (not one per dimension).
template <typename T, int DIM>
struct CoordRec {
  static constexpr int PACK = DIM == 3 ? 4 : DIM;
  static __device__ __forceinline__ void store(T *rec, const T (&v)[DIM]) {
    if constexpr (DIM == 1) {
      rec[0] = v[0];
    } else if constexpr (DIM == 2) {
      using V2 = typename std::conditional<std::is_same<T, float>::value, float2, double2>::type;
      *reinterpret_cast<V2 *>(rec) = V2{v[0], v[1]};
    } else if constexpr (std::is_same<T, float>::value) {
      *reinterpret_cast<float4 *>(rec) = make_float4(v[0], v[1], v[2], 0.f);
    } else {
      reinterpret_cast<double2 *>(rec)[0] = make_double2(v[0], v[1]);
      reinterpret_cast<double2 *>(rec)[1] = make_double2(v[2], 0.0);
    }
  }
  static __device__ __forceinline__ void load(const T *rec, T (&v)[DIM]) {
    if constexpr (DIM == 1) {
      v[0] = rec[0];
    } else if constexpr (DIM == 2) {
      using V2 = typename std::conditional<std::is_same<T, float>::value, float2, double2>::type;
      const V2 t = *reinterpret_cast<const V2 *>(rec);
      v[0] = t.x;
      v[1] = t.y;
    } else if constexpr (std::is_same<T, float>::value) {
      const float4 t = *reinterpret_cast<const float4 *>(rec);
      v[0] = t.x;
      v[1] = t.y;
      v[2] = t.z;
    } else {
      const double2 t0 = reinterpret_cast<const double2 *>(rec)[0];
      const double2 t1 = reinterpret_cast<const double2 *>(rec)[1];
      v[0] = t0.x;
      v[1] = t0.y;
      v[2] = t1.x;
    }
  }
};

__device__ __forceinline__ float above(float v) { return nextafterf(v, INFINITY); }
__device__ __forceinline__ double above(double v) { return ::nextafter(v, (double)INFINITY); }

// Key and bin-relative coordinates of point j (see cell_count_kernel).
// ORIGIN false: the point is binned by its cell floor(g).  ORIGIN true: by
// the node q = ceil(g - oc) mod n (oc = 1/2 for odd w, 0 for even w), which
// is ceil(g - w/2) + floor(w/2), the first node of its support shifted by
// floor(w/2); its bin-relative coordinate v is then kept in (q_rel - 1 + oc,
// q_rel + oc], where ceil(v - w/2) + floor(w/2) = q_rel, and is taken one
// period down when q wrapped from n to 0.
template <typename T, int DIM, bool ORIGIN>
__device__ __forceinline__ int32_t cell_key(const PointsIn &a, int64_t j, T (&out)[DIM], bool *bad) {
  int bin = 0, stride = 1, local = 0, lstride = 1;
#pragma unroll
  for (int d = 0; d < DIM; d++) {
    int cell = 0;
    T v = T(0);
    bool done = false;
    if constexpr (std::is_same<T, float>::value) {
      float gh, gl, delta;
      if (a.fast && fold_fast_hl(static_cast<const float *>(a.x[d])[j], a.turn3, a.n[d], &gh, &gl, &delta)) {
        if constexpr (!ORIGIN) {
          if (cell_from_hl(gh, gl, delta, a.n[d], &cell)) {
            v = (gh - (float)((cell / a.m[d]) * a.m[d])) + gl;  // the difference is exact
            done = true;
          }
        } else if (node_from_hl(gh, gl, delta, a.oc, a.n[d], &cell)) {
          const float hw = cell == a.n[d] ? gh - (float)a.n[d] : gh;  // exact
          if (cell == a.n[d]) cell = 0;
          v = (hw - (float)((cell / a.m[d]) * a.m[d])) + gl;
          done = true;
        }
      }
    }
    if (!done) {
      double g = grid_coord(load_coord<T>(a.x[d], j), a.inv_two_pi, a.n[d], bad);
      if constexpr (!ORIGIN) {
        cell = (int)floor(g);
        if (cell >= a.n[d]) cell = a.n[d] - 1;  // unreachable; keeps the index in range
      } else {
        cell = (int)ceil(g - (double)a.oc);
        if (cell >= a.n[d]) {
          cell = 0;
          g -= (double)a.n[d];
        }
      }
      v = (T)(g - (double)((cell / a.m[d]) * a.m[d]));  // exact in double, then rounded to T
    }
    const int b = cell / a.m[d];
    const int cell_rel = cell - b * a.m[d];
    bin += b * stride;
    stride *= a.nb[d];
    local += cell_rel * lstride;
    lstride *= a.m[d];
    if constexpr (!ORIGIN) {
      if (floor(v) > (T)cell_rel) v = below(T(cell_rel + 1));
      if (v < (T)cell_rel) v = (T)cell_rel;
    } else {
      const T hi_v = (T)cell_rel + (T)a.oc;
      if (v > hi_v) v = hi_v;
      if (v <= hi_v - T(1)) v = above(hi_v - T(1));
    }
    out[d] = v;
  }
  return bin * lstride + local;
}

// Cell-level key of a point: its bin, then its cell inside the bin (x fastest).
// Sorting by this key orders the points bin by bin (as Sec. III-A) and, inside
// each bin, cell by cell, so a bin's points of one fine-grid row (and one x
// range of that row) form a contiguous run.
// The fold to the fine grid is done once, here: the point's bin-relative
// coordinate, rounded to T but never up to the next cell (floor stays the
// point's cell), is written in the caller's order, one record per point
// (CoordRec), and later gathered into sorted order.  Each thread takes PPT
// points blockDim.x apart and issues their counter increments back to back,
// so that several returning atomics are in flight per thread.
template <typename T, int DIM, int PPT, bool ORIGIN>
__global__ void cell_count_kernel(PointsIn a, int32_t *counts, int32_t *key_of, int32_t *rank_of,
                                  int *flag, T *rel) {
  using R = CoordRec<T, DIM>;
  const int64_t j0 = (int64_t)blockIdx.x * blockDim.x * PPT + threadIdx.x;
  bool bad = false;
  int32_t key[PPT];
#pragma unroll
  for (int u = 0; u < PPT; u++) {
    const int64_t j = j0 + (int64_t)u * blockDim.x;
    key[u] = 0;
    if (j < a.M) {
      T v[DIM];
      key[u] = cell_key<T, DIM, ORIGIN>(a, j, v, &bad);
      R::store(rel + j * R::PACK, v);
    }
  }
  int32_t rank[PPT];
#pragma unroll
  for (int u = 0; u < PPT; u++)
    if (j0 + (int64_t)u * blockDim.x < a.M) rank[u] = atomicAdd(&counts[key[u]], 1);
#pragma unroll
  for (int u = 0; u < PPT; u++) {
    const int64_t j = j0 + (int64_t)u * blockDim.x;
    if (j < a.M) {
      key_of[j] = key[u];
      rank_of[j] = rank[u];
    }
  }
  if (bad) atomicOr(flag, 1);
}

// Sorted slot of each point: the one scattered store of the sort.  PPT
// points per thread, blockDim.x apart, with their loads issued together.
template <int PPT>
__global__ void cell_scatter_kernel(int64_t M, const int32_t *starts, const int32_t *key_of,
                                    const int32_t *rank_of, int32_t *perm) {
  const int64_t j0 = (int64_t)blockIdx.x * blockDim.x * PPT + threadIdx.x;
  int32_t key[PPT], rank[PPT], slot[PPT];
#pragma unroll
  for (int u = 0; u < PPT; u++) {
    const int64_t j = j0 + (int64_t)u * blockDim.x;
    key[u] = j < M ? key_of[j] : 0;
    rank[u] = j < M ? rank_of[j] : 0;
  }
#pragma unroll
  for (int u = 0; u < PPT; u++) slot[u] = j0 + (int64_t)u * blockDim.x < M ? starts[key[u]] + rank[u] : 0;
#pragma unroll
  for (int u = 0; u < PPT; u++) {
    const int64_t j = j0 + (int64_t)u * blockDim.x;
    if (j < M) perm[slot[u]] = (int32_t)j;
  }
}

// Bin-relative coordinates in sorted order: coalesced writes, one record per
// point gathered through the permutation.  PPT slots per thread, blockDim.x
// apart.
template <typename T, int DIM, int PPT>
__global__ void gather_coords_kernel(int64_t M, const int32_t *perm, const T *rel, T *g0, T *g1, T *g2) {
  using R = CoordRec<T, DIM>;
  const int64_t q0 = (int64_t)blockIdx.x * blockDim.x * PPT + threadIdx.x;
  int32_t src[PPT];
#pragma unroll
  for (int u = 0; u < PPT; u++) {
    const int64_t q = q0 + (int64_t)u * blockDim.x;
    src[u] = q < M ? perm[q] : 0;
  }
  T v[PPT][DIM];
#pragma unroll
  for (int u = 0; u < PPT; u++)
    if (q0 + (int64_t)u * blockDim.x < M) R::load(rel + (int64_t)src[u] * R::PACK, v[u]);
  T *const g[3] = {g0, g1, g2};
#pragma unroll
  for (int u = 0; u < PPT; u++) {
    const int64_t q = q0 + (int64_t)u * blockDim.x;
    if (q < M) {
#pragma unroll
      for (int d = 0; d < DIM; d++) g[d][q] = v[u][d];
    }
  }
}

// Bin counts and starts from the cell starts (cpb cells per bin).
__global__ void bins_from_cells_kernel(const int32_t *cell_starts, int64_t nbins, int64_t cpb,
                                       int32_t *counts, int32_t *starts) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b > nbins) return;
  const int32_t s0 = cell_starts[b * cpb];
  starts[b] = s0;
  if (b < nbins) counts[b] = cell_starts[(b + 1) * cpb] - s0;
}

// GM (no sort): each point's fine-grid cell, packed l1 + n1 (l2 + n2 l3), and
// its offset inside the cell, in the caller's order.
template <typename T>
__global__ void gm_prepare_kernel(PointsIn a, int32_t *packed, T *f0, T *f1, T *f2, int *flag) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= a.M) return;
  T *out[3] = {f0, f1, f2};
  bool bad = false;
  int64_t cell_index = 0, stride = 1;
  for (int d = 0; d < a.dim; d++) {
    double g = grid_coord(load_coord<T>(a.x[d], j), a.inv_two_pi, a.n[d], &bad);
    int cell = (int)floor(g);
    if (cell >= a.n[d]) cell = a.n[d] - 1;
    T v = (T)(g - (double)cell);  // exact in double, then rounded to T
    if (v >= T(1)) v = below(T(1));
    out[d][j] = v;
    cell_index += (int64_t)cell * stride;
    stride *= a.n[d];
  }
  if (bad) atomicOr(flag, 1);
  packed[j] = (int32_t)cell_index;
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
  e.groups = 0;
  table[s] = e;
}

// inv_two_pi = c0 + c1 + c2 exactly: c0 its nearest float, c1 the nearest
// float to the (exact) remainder, c2 the rest, which has at most 53 - 48
// significant bits and so is a float too.
void split_turn(PointsIn &a) {
  const double c = a.inv_two_pi;
  const float c0 = (float)c;
  const double r = c - (double)c0;
  const float c1 = (float)r;
  const float c2 = (float)(r - (double)c1);
  a.turn3[0] = c0;
  a.turn3[1] = c1;
  a.turn3[2] = c2;
  a.fast = ((double)c0 + (double)c1) + (double)c2 == c;
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

template <typename T, int PPT>
cudaError_t launch_cell_count(int dim, unsigned blocks, int threads, cudaStream_t s, const PointsIn &a,
                              nufft_plan_s *p) {
  T *rel = static_cast<T *>(p->gtmp);
  if (dim == 1)
    cell_count_kernel<T, 1, PPT, false><<<blocks, threads, 0, s>>>(a, p->cell_counts, p->bin_of, p->rank_of,
                                                                   p->flag, rel);
  else if (dim == 2)
    cell_count_kernel<T, 2, PPT, false><<<blocks, threads, 0, s>>>(a, p->cell_counts, p->bin_of, p->rank_of,
                                                                   p->flag, rel);
  else if (!a.origin)
    cell_count_kernel<T, 3, PPT, false><<<blocks, threads, 0, s>>>(a, p->cell_counts, p->bin_of, p->rank_of,
                                                                   p->flag, rel);
  else
    cell_count_kernel<T, 3, PPT, true><<<blocks, threads, 0, s>>>(a, p->cell_counts, p->bin_of, p->rank_of,
                                                                  p->flag, rel);
  return cudaGetLastError();
}

template <typename T, int PPT>
cudaError_t launch_gather_coords(int dim, unsigned blocks, int threads, cudaStream_t s, int64_t M,
                                 nufft_plan_s *p) {
  const T *rel = static_cast<const T *>(p->gtmp);
  T *g0 = static_cast<T *>(p->gcoord[0]);
  T *g1 = static_cast<T *>(dim >= 2 ? p->gcoord[1] : p->gcoord[0]);
  T *g2 = static_cast<T *>(dim == 3 ? p->gcoord[2] : p->gcoord[0]);
  if (dim == 1)
    gather_coords_kernel<T, 1, PPT><<<blocks, threads, 0, s>>>(M, p->perm, rel, g0, g1, g2);
  else if (dim == 2)
    gather_coords_kernel<T, 2, PPT><<<blocks, threads, 0, s>>>(M, p->perm, rel, g0, g1, g2);
  else
    gather_coords_kernel<T, 3, PPT><<<blocks, threads, 0, s>>>(M, p->perm, rel, g0, g1, g2);
  return cudaGetLastError();
}

}  // namespace

int run_setpts(nufft_plan_s *p, const void *x, const void *y, const void *z) {
  const int64_t M = p->M;
  cudaStream_t s = p->stream;
  const size_t rs = real_size(p);
  const int64_t cpb = (int64_t)p->m[0] * p->m[1] * p->m[2];  // cells per bin
  const int64_t nkeys = p->nbins * cpb;

  // --- storage (grown, never shrunk) --------------------------------------
  if (p->nbins + 1 > p->cap_bins || !p->bin_counts) {
    cudaFree(p->bin_counts);
    cudaFree(p->bin_starts);
    cudaFree(p->sub_counts);
    cudaFree(p->sub_starts);
    p->bin_counts = p->bin_starts = p->sub_counts = p->sub_starts = nullptr;
    p->cap_bins = 0;
    const size_t nb = (size_t)(p->nbins + 1) * sizeof(int32_t);
    if (cudaMalloc((void **)&p->bin_counts, nb) != cudaSuccess ||
        cudaMalloc((void **)&p->bin_starts, nb) != cudaSuccess ||
        cudaMalloc((void **)&p->sub_counts, nb) != cudaSuccess ||
        cudaMalloc((void **)&p->sub_starts, nb) != cudaSuccess)
      return NUFFT_ERR_ALLOC;
    p->cap_bins = p->nbins + 1;
  }
  if (nkeys + 1 > p->cap_keys || !p->cell_counts) {
    cudaFree(p->cell_counts);
    cudaFree(p->cell_starts);
    cudaFree(p->scan_scratch);
    p->cell_counts = p->cell_starts = p->scan_scratch = nullptr;
    p->cap_keys = 0;
    const size_t nk = (size_t)(nkeys + 1) * sizeof(int32_t);
    if (cudaMalloc((void **)&p->cell_counts, nk) != cudaSuccess ||
        cudaMalloc((void **)&p->cell_starts, nk) != cudaSuccess ||
        cudaMalloc((void **)&p->scan_scratch,
                   (size_t)scan_scratch_len(nkeys + 1) * sizeof(int32_t)) != cudaSuccess)
      return NUFFT_ERR_ALLOC;
    p->cap_keys = nkeys + 1;
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
  // caller-order bin-relative coordinates (dim arrays of M reals)
  const int pack = p->dim == 3 ? 4 : p->dim;  // CoordRec<T, dim>::PACK
  if (grow(&p->gtmp, &p->cap_gtmp, (int64_t)pack * (M > 0 ? M : 1), rs) != cudaSuccess)
    return NUFFT_ERR_ALLOC;

  // --- 1. cells, bins and counts ------------------------------------------
  PointsIn a{};
  a.x[0] = x;
  a.x[1] = y;
  a.x[2] = p->dim == 3 ? z : x;
  a.M = M;
  a.dim = p->dim;
  a.is_double = p->dtype;
  a.inv_two_pi = 1.0 / (2.0 * 3.14159265358979323846);
  split_turn(a);
  a.origin = p->bin_origin ? 1 : 0;
  a.oc = p->w % 2 ? 0.5f : 0.0f;
  for (int d = 0; d < 3; d++) {
    a.n[d] = (int)p->n[d];
    a.m[d] = p->m[d];
    a.nb[d] = p->nb[d];
  }
  if (cudaMemsetAsync(p->cell_counts, 0, (size_t)(nkeys + 1) * 4, s) != cudaSuccess ||
      cudaMemsetAsync(p->flag, 0, sizeof(int), s) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  const int threads = 256;
  if (M > 0) {
    constexpr int kPPT = 4;
    const unsigned blocks_cc = (unsigned)((M + threads * kPPT - 1) / (threads * kPPT));
    const cudaError_t e = p->dtype == 0 ? launch_cell_count<float, kPPT>(p->dim, blocks_cc, threads, s, a, p)
                                        : launch_cell_count<double, kPPT>(p->dim, blocks_cc, threads, s, a, p);
    if (e != cudaSuccess) return NUFFT_ERR_CUDA;
  }

  // --- 2. cell starts (bin starts are every cpb-th entry) -----------------
  if (exclusive_scan(p->cell_counts, p->cell_starts, nkeys, p->scan_scratch, s) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  const unsigned blocks_bins = (unsigned)((p->nbins + 1 + threads - 1) / threads);
  bins_from_cells_kernel<<<blocks_bins, threads, 0, s>>>(p->cell_starts, p->nbins, cpb,
                                                         p->bin_counts, p->bin_starts);
  if (cudaGetLastError() != cudaSuccess) return NUFFT_ERR_CUDA;

  // --- 3. permutation and sorted coordinates ------------------------------
  if (M > 0) {
    constexpr int kPPT = 4;
    const unsigned blocks_ppt = (unsigned)((M + threads * kPPT - 1) / (threads * kPPT));
    cell_scatter_kernel<kPPT><<<blocks_ppt, threads, 0, s>>>(M, p->cell_starts, p->bin_of, p->rank_of, p->perm);
    if ((p->dtype == 0 ? launch_gather_coords<float, kPPT>(p->dim, blocks_ppt, threads, s, M, p)
                       : launch_gather_coords<double, kPPT>(p->dim, blocks_ppt, threads, s, M, p)) != cudaSuccess)
      return NUFFT_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return NUFFT_ERR_CUDA;
  }

  // --- 4. subproblems ------------------------------------------------------
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

  // --- 5. window-origin groups of the grouped 3D interpolator -------------
  if (p->igroup >= 2) {
    if (grow(&p->grec, &p->cap_grec, M > 0 ? M : 1, sizeof(uint32_t)) != cudaSuccess) return NUFFT_ERR_ALLOC;
    if (build_groups3d(p) != cudaSuccess) return NUFFT_ERR_CUDA;
  }
  return NUFFT_OK;
}

// GM setpts: no bin sort, only the per-point cell and offset.
int run_setpts_gm(nufft_plan_s *p, const void *x, const void *y, const void *z) {
  const int64_t M = p->M;
  cudaStream_t s = p->stream;
  const size_t rs = real_size(p);
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
  PointsIn a{};
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
  if (cudaMemsetAsync(p->flag, 0, sizeof(int), s) != cudaSuccess) return NUFFT_ERR_CUDA;
  const int threads = 256;
  if (M > 0) {
    const unsigned blocks = (unsigned)((M + threads - 1) / threads);
    if (p->dtype == 0)
      gm_prepare_kernel<float><<<blocks, threads, 0, s>>>(
          a, p->bin_of, (float *)p->gcoord[0], (float *)p->gcoord[1],
          (float *)(p->dim == 3 ? p->gcoord[2] : p->gcoord[0]), p->flag);
    else
      gm_prepare_kernel<double><<<blocks, threads, 0, s>>>(
          a, p->bin_of, (double *)p->gcoord[0], (double *)p->gcoord[1],
          (double *)(p->dim == 3 ? p->gcoord[2] : p->gcoord[0]), p->flag);
    if (cudaGetLastError() != cudaSuccess) return NUFFT_ERR_CUDA;
  }
  int host_flag = 0;
  if (cudaMemcpyAsync(&host_flag, p->flag, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  if (host_flag) return NUFFT_ERR_BAD_POINTS;
  p->nsub = 0;
  p->nbins = 0;
  return NUFFT_OK;
}

}  // namespace nufft

namespace nufft {
// ===================================================================== no-allocation bin sort
//
// nufft_binsort_noalloc: the bin sort above (count, scan, permute) for callers
// that must not allocate device memory.  Its scratch (each point's bin and
// rank, the bin starts, the scan partials, the error flag) lives in the
// file-scope array below instead of cudaMalloc'd buffers.

namespace {

constexpr int64_t kNoAllocMaxPoints = int64_t(1) << 20;  // 1,048,576 points
constexpr int64_t kNoAllocMaxBins = int64_t(1) << 16;    // 65,536 bins

constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
constexpr size_t kOffBinOf = 0;
constexpr size_t kOffRankOf = align256(kOffBinOf + sizeof(int32_t) * kNoAllocMaxPoints);
constexpr size_t kOffStarts = align256(kOffRankOf + sizeof(int32_t) * kNoAllocMaxPoints);
constexpr size_t kOffScan = align256(kOffStarts + sizeof(int32_t) * (kNoAllocMaxBins + 1));
constexpr size_t kScanInts = (kNoAllocMaxBins + 1 + 4095) / 4096 + 1;  // scan_scratch_len bound
constexpr size_t kOffFlag = align256(kOffScan + sizeof(int32_t) * kScanInts);
constexpr size_t kNoAllocBytes = align256(kOffFlag + sizeof(int));  // about 8.3 MB

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
unsigned char *g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
int noalloc_scratch(unsigned char **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NUFFT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return NUFFT_ERR_CUDA;
    }
    g_noalloc_addr[dev] = static_cast<unsigned char *>(p);
  }
  *out = g_noalloc_addr[dev];
  return NUFFT_OK;
}

// Writes only the permutation: slot starts[bin] + rank <- caller index.
__global__ void permute_only_kernel(int64_t M, const int32_t *starts, const int32_t *bin_of,
                                    const int32_t *rank_of, int32_t *perm) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= M) return;
  perm[starts[bin_of[j]] + rank_of[j]] = (int32_t)j;
}

}  // namespace
}  // namespace nufft

using nufft::PointsIn;

extern "C" int nufft_binsort_noalloc(int dim, int dtype, int64_t M, const void *x, const void *y,
                                     const void *z, const int64_t *n_fine, const int64_t *bins,
                                     int32_t *counts, int32_t *perm, void *cuda_stream) {
  if ((dim != 2 && dim != 3) || (dtype != 0 && dtype != 1) || M < 0 || !n_fine || !bins ||
      !counts || (M > 0 && (!x || !y || (dim == 3 && !z) || !perm)))
    return NUFFT_ERR_BAD_ARG;
  PointsIn a{};
  for (int d = 0; d < 3; d++) {
    const int64_t n = d < dim ? n_fine[d] : 1, m = d < dim ? bins[d] : 1;
    if (n < 1 || m < 1 || n > (int64_t(1) << 30)) return NUFFT_ERR_BAD_ARG;
    a.n[d] = (int)n;
    a.m[d] = (int)(m < n ? m : n);
    a.nb[d] = (int)((n + a.m[d] - 1) / a.m[d]);
  }
  if (M > nufft::kNoAllocMaxPoints) return NUFFT_ERR_TOO_LARGE;
  // bins per dimension can reach 2^30 each: test each factor against the
  // limit before multiplying, so the product never overflows
  int64_t nbins = 1;
  for (int d = 0; d < 3; d++) {
    if (a.nb[d] > nufft::kNoAllocMaxBins / nbins) return NUFFT_ERR_TOO_LARGE;
    nbins *= a.nb[d];
  }
  unsigned char *base = nullptr;
  int rc = nufft::noalloc_scratch(&base);
  if (rc) return rc;
  using namespace nufft;
  int32_t *bin_of = reinterpret_cast<int32_t *>(base + kOffBinOf);
  int32_t *rank_of = reinterpret_cast<int32_t *>(base + kOffRankOf);
  int32_t *starts = reinterpret_cast<int32_t *>(base + kOffStarts);
  int32_t *scan = reinterpret_cast<int32_t *>(base + kOffScan);
  int *flag = reinterpret_cast<int *>(base + kOffFlag);
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

  a.x[0] = x;
  a.x[1] = y;
  a.x[2] = dim == 3 ? z : x;
  a.M = M;
  a.dim = dim;
  a.is_double = dtype;
  a.inv_two_pi = 1.0 / (2.0 * 3.14159265358979323846);
  // the shared scratch keeps the previous call's contents: clear what sums
  if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)nbins, s) != cudaSuccess ||
      cudaMemsetAsync(flag, 0, sizeof(int), s) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  const int threads = 256;
  const unsigned blocks = (unsigned)((M + threads - 1) / threads);
  if (M > 0) {
    if (dtype == 0)
      nufft::bin_count_kernel<float><<<blocks, threads, 0, s>>>(a, counts, bin_of, rank_of, flag);
    else
      nufft::bin_count_kernel<double><<<blocks, threads, 0, s>>>(a, counts, bin_of, rank_of, flag);
    if (cudaGetLastError() != cudaSuccess) return NUFFT_ERR_CUDA;
  }
  if (nufft::exclusive_scan(counts, starts, nbins, scan, s) != cudaSuccess) return NUFFT_ERR_CUDA;
  if (M > 0) {
    nufft::permute_only_kernel<<<blocks, threads, 0, s>>>(M, starts, bin_of, rank_of, perm);
    if (cudaGetLastError() != cudaSuccess) return NUFFT_ERR_CUDA;
  }
  int host_flag = 0;
  if (cudaMemcpyAsync(&host_flag, flag, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  return host_flag ? NUFFT_ERR_BAD_POINTS : NUFFT_OK;
}
