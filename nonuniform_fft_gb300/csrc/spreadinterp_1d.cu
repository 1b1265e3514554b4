// 1D spreading and interpolation.
//
// "cuFINUFFT: a load-balanced GPU library for general-purpose nonuniform
// FFTs" defines the transforms in 2D and notes that the definitions
// generalize to 1D in the obvious fashion (Sec. I); the steps of Sec. II then
// read, in 1D: spreading b_l = sum_j c_j psi_per(l h - x_j) (eq. (7)), and
// interpolation c_j = sum_l b_l psi_per(l h - x_j) (Sec. II-B c).
//   * Spreading uses the same decomposition as in 2D: bins of
//     32 - 2 ceil(w/2) cells, subproblems of at most M_sub cell-sorted points,
//     one warp per subproblem, lane L owning padded-bin column L.  A lane
//     visits the points of the cells whose support reaches its column (a
//     contiguous run of the sorted points), evaluates the kernel for its own
//     node and accumulates in a register; at the end each lane adds its
//     column into the fine grid (eq. (15)).
//   * Interpolation: one block per subproblem stages the padded bin of the
//     fine grid in shared memory, one thread per point reads its w nodes.
#include <type_traits>

#include "spread_regtile.cuh"

namespace nufft {
namespace {

template <typename T>
struct Params1D {
  using CT = typename Cplx<T>::type;
  const Subproblem *sub;
  int nsub;
  const int32_t *perm;
  const T *g1;                 // bin-relative coordinate in cells
  const int32_t *cell_starts;  // per (bin, cell)
  const CT *c_in;
  CT *c_out;
  CT *grid;
  T beta_e;
  int n1, m1;
  int64_t cstride, gstride;  // per vector: M strengths, one fine grid
};

constexpr int kWarps1D = 4;

template <typename T, int W>
__global__ void __launch_bounds__(32 * kWarps1D) spread_reg1d_kernel(Params1D<T> a) {
  using CT = typename Cplx<T>::type;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_in += blockIdx.y * a.cstride;
  constexpr int PAD = (W + 1) / 2, HW = W / 2, S = 128;
  __shared__ T s_g[kWarps1D][S];
  __shared__ CT s_c[kWarps1D][S];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sidx = blockIdx.x * kWarps1D + warp;
  if (sidx >= a.nsub) return;  // whole warp leaves together
  const Subproblem sp = a.sub[sidx];
  const int lo = sp.start, hi = sp.start + sp.count;
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int32_t *cs = a.cell_starts + (int64_t)sp.bin * a.m1;
  // column x_rel = lane - PAD takes points whose cell lies in [x_rel + HW - W, x_rel + HW]
  const int x_rel = lane - PAD;
  int xw_lo = x_rel + HW - W, xw_hi = x_rel + HW + 1;
  xw_lo = xw_lo < 0 ? 0 : xw_lo;
  xw_hi = xw_hi > a.m1 ? a.m1 : xw_hi;
  int llo = hi, lhi = hi;
  if (xw_lo < xw_hi) {
    llo = cs[xw_lo] > lo ? cs[xw_lo] : lo;
    lhi = cs[xw_hi] < hi ? cs[xw_hi] : hi;
  }
  const T scale = T(2) / T(W);
  T ar = T(0), ai = T(0);
  for (int bs = lo; bs < hi; bs += S) {
    const int nb = (bs + S < hi ? bs + S : hi) - bs;
    for (int q = lane; q < nb; q += 32) {
      s_g[warp][q] = ld_hint(a.g1 + bs + q, pol_stream);
      s_c[warp][q] = ld_hint(a.c_in + ld_hint(a.perm + bs + q, pol_stream), pol_keep);
    }
    __syncwarp();
    const int j0 = llo > bs ? llo : bs, j1 = lhi < bs + nb ? lhi : bs + nb;
    for (int j = j0; j < j1; j++) {
      const T g = s_g[warp][j - bs];
      // this column is one of the point's w nodes l0 .. l0 + w - 1, l0 = ceil(g - w/2)
      const int t = x_rel - (int)es_ceil(g - T(0.5) * T(W));
      const T wt = (t >= 0 && t < W) ? es_fast((T(x_rel) - g) * scale, a.beta_e) : T(0);
      const CT cv = s_c[warp][j - bs];
      ar += cv.x * wt;
      ai += cv.y * wt;
    }
    __syncwarp();
  }
  if (ar != T(0) || ai != T(0))
    grid_atomic_add(a.grid + wrap_tile(sp.bin * a.m1 + x_rel, a.n1), ar, ai);
}

// A complex two-float, 16-byte aligned so that it moves as one 16-byte
// shared-memory access.
struct __align__(16) DFC16 {
  DF re, im;
};

// Double precision: each point's w+1 extended kernel values are evaluated
// once, in two-float arithmetic (df64.cuh), when its batch is staged, and
// stored as two-float products c_j phi; a lane-visit is then one 16-byte
// load and two two-float adds.  Only the coordinate split and the final
// column sum touch the FP64 pipe, which this part runs at 1/64 of the FP32
// rate (native double products and sums per slot and per lane-visit kept it
// busy 84 % of the time and took 1.48 ms on the 1D workload).
template <int W>
__global__ void __launch_bounds__(32 * kWarps1D) spread_reg1d_df_kernel(Params1D<double> a) {
  constexpr int PAD = (W + 1) / 2, HW = W / 2, WX = W + 1, WCS = WX | 1;
  constexpr int S = W <= 8 ? 64 : 32;
  __shared__ DFC16 s_cw[kWarps1D][S][WCS];
  __shared__ int s_xb[kWarps1D][S];
  __shared__ DF s_exp2[64];
  fill_exp2_64(s_exp2);
  __syncthreads();
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_in += blockIdx.y * a.cstride;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sidx = blockIdx.x * kWarps1D + warp;
  if (sidx >= a.nsub) return;  // whole warp leaves together
  const Subproblem sp = a.sub[sidx];
  const int lo = sp.start, hi = sp.start + sp.count;
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int32_t *cs = a.cell_starts + (int64_t)sp.bin * a.m1;
  const int x_rel = lane - PAD;
  int xw_lo = x_rel + HW - W, xw_hi = x_rel + HW + 1;
  xw_lo = xw_lo < 0 ? 0 : xw_lo;
  xw_hi = xw_hi > a.m1 ? a.m1 : xw_hi;
  int llo = hi, lhi = hi;
  if (xw_lo < xw_hi) {
    llo = cs[xw_lo] > lo ? cs[xw_lo] : lo;
    lhi = cs[xw_hi] < hi ? cs[xw_hi] : hi;
  }
  const DF beta = df_from(a.beta_e);
  DF ar{0.f, 0.f}, ai{0.f, 0.f};
  for (int bs = lo; bs < hi; bs += S) {
    const int nb = (bs + S < hi ? bs + S : hi) - bs;
    for (int q = lane; q < nb; q += 32) {
      const double2 cv = ld_hint(a.c_in + ld_hint(a.perm + bs + q, pol_stream), pol_keep);
      DF ext[WX];
      s_xb[warp][q] = es_extended_df<W, WX>(ld_hint(a.g1 + bs + q, pol_stream), beta, ext, s_exp2);
      const DF cr = df_from(cv.x), ci = df_from(cv.y);
#pragma unroll
      for (int e = 0; e < WX; e++) {
        DFC16 v;
        v.re = df_mul(cr, ext[e]);
        v.im = df_mul(ci, ext[e]);
        s_cw[warp][q][e] = v;
      }
    }
    __syncwarp();
    const int j0 = llo > bs ? llo : bs, j1 = lhi < bs + nb ? lhi : bs + nb;
    for (int j = j0; j < j1; j++) {
      const int q = j - bs;
      int e = x_rel - s_xb[warp][q];
      e = e < 0 ? 0 : (e > W ? W : e);
      const DFC16 v = s_cw[warp][q][e];
      ar = df_sum(ar, v.re);
      ai = df_sum(ai, v.im);
    }
    __syncwarp();
  }
  const double vr = df_to(ar), vi = df_to(ai);
  if (vr != 0.0 || vi != 0.0) grid_atomic_add(a.grid + wrap_tile(sp.bin * a.m1 + x_rel, a.n1), vr, vi);
}

// Single precision (double: interp_sm1d_df_kernel below).
template <typename T, int W>
__global__ void interp_sm1d_kernel(Params1D<T> a) {
  using CT = typename Cplx<T>::type;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_out += blockIdx.y * a.cstride;
  constexpr int PAD = (W + 1) / 2;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  CT *tile = reinterpret_cast<CT *>(smem_raw);
  const Subproblem sp = a.sub[blockIdx.x];
  const int p1 = a.m1 + 2 * PAD;
  const int o1 = sp.bin * a.m1 - PAD;
  for (int s = threadIdx.x; s < p1; s += blockDim.x) tile[s] = a.grid[wrap_tile(o1 + s, a.n1)];
  __syncthreads();
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int end = sp.start + sp.count;
  for (int j = sp.start + threadIdx.x; j < end; j += blockDim.x) {
    T k1[W];
    const int s1 = es_weights<T, W>(ld_hint(a.g1 + j, pol_stream), a.beta_e, k1) + PAD;
    T ar = T(0), ai = T(0);
#pragma unroll
    for (int i1 = 0; i1 < W; i1++) {
      const CT b = tile[s1 + i1];
      ar += b.x * k1[i1];
      ai += b.y * k1[i1];
    }
    CT out;
    out.x = ar;
    out.y = ai;
    st_hint(a.c_out + ld_hint(a.perm + j, pol_stream), out, pol_keep);
  }
}

// Double precision: the padded bin is staged as two-floats and the w
// multiply-adds run in two-float arithmetic on the FP32 pipes (df64.cuh);
// the kernel values come from the same two-float evaluation as the
// spreader's.  At most 16 terms: accumulated without renormalisation
// (df_fma_lazy), the sum hi + lo converted to double exactly.
template <int W>
__global__ void interp_sm1d_df_kernel(Params1D<double> a) {
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_out += blockIdx.y * a.cstride;
  constexpr int PAD = (W + 1) / 2;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  DFC16 *tile = reinterpret_cast<DFC16 *>(smem_raw);
  __shared__ DF s_exp2[64];
  fill_exp2_64(s_exp2);
  const Subproblem sp = a.sub[blockIdx.x];
  const int p1 = a.m1 + 2 * PAD;
  const int o1 = sp.bin * a.m1 - PAD;
  for (int s = threadIdx.x; s < p1; s += blockDim.x) {
    const double2 v = a.grid[wrap_tile(o1 + s, a.n1)];
    DFC16 d;
    d.re = df_from(v.x);
    d.im = df_from(v.y);
    tile[s] = d;
  }
  __syncthreads();
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const DF beta = df_from(a.beta_e);
  const int end = sp.start + sp.count;
  for (int j = sp.start + threadIdx.x; j < end; j += blockDim.x) {
    DF k1[W];
    const int s1 = es_weights_df<W>(ld_hint(a.g1 + j, pol_stream), beta, k1, s_exp2) + PAD;
    DF ar{0.f, 0.f}, ai{0.f, 0.f};
#pragma unroll
    for (int i1 = 0; i1 < W; i1++) {
      const DFC16 b = tile[s1 + i1];
      df_fma_lazy(ar, b.re, k1[i1]);
      df_fma_lazy(ai, b.im, k1[i1]);
    }
    double2 out;
    out.x = df_to(ar);
    out.y = df_to(ai);
    st_hint(a.c_out + ld_hint(a.perm + j, pol_stream), out, pol_keep);
  }
}

template <typename T>
Params1D<T> params1d(const nufft_plan_s *p) {
  Params1D<T> a{};
  a.sub = p->subprob;
  a.nsub = (int)p->nsub;
  a.perm = p->perm;
  a.g1 = static_cast<const T *>(p->gcoord[0]);
  a.cell_starts = p->cell_starts;
  a.c_in = nullptr;
  a.c_out = nullptr;
  a.grid = static_cast<typename Cplx<T>::type *>(p->grid);
  a.beta_e = (T)es_beta_e(p->beta, sizeof(T));
  a.n1 = (int)p->n[0];
  a.m1 = p->m[0];
  a.cstride = p->M;
  a.gstride = grid_cells(p);
  return a;
}

template <typename T, int W>
cudaError_t spread1d_w(const nufft_plan_s *p, const void *c) {
  Params1D<T> a = params1d<T>(p);
  a.c_in = static_cast<const typename Cplx<T>::type *>(c);
  const dim3 grid((unsigned)((p->nsub + kWarps1D - 1) / kWarps1D), p->nvec);
  if constexpr (std::is_same<T, double>::value)
    spread_reg1d_df_kernel<W><<<grid, 32 * kWarps1D, 0, p->stream>>>(a);
  else
    spread_reg1d_kernel<T, W><<<grid, 32 * kWarps1D, 0, p->stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int W>
cudaError_t interp1d_w(const nufft_plan_s *p, void *c) {
  Params1D<T> a = params1d<T>(p);
  a.c_out = static_cast<typename Cplx<T>::type *>(c);
  if constexpr (std::is_same<T, double>::value) {
    const size_t smem = (size_t)(p->m[0] + 2 * ((W + 1) / 2)) * sizeof(DFC16);
    cudaError_t e = allow_smem(interp_sm1d_df_kernel<W>, smem);
    if (e != cudaSuccess) return e;
    interp_sm1d_df_kernel<W><<<dim3((unsigned)p->nsub, p->nvec), block_threads(interp_sm1d_df_kernel<W>, p->threads),
                               smem, p->stream>>>(a);
    return cudaGetLastError();
  } else {
    const size_t smem = (size_t)(p->m[0] + 2 * ((W + 1) / 2)) * 2 * sizeof(T);
    cudaError_t e = allow_smem(interp_sm1d_kernel<T, W>, smem);
    if (e != cudaSuccess) return e;
    interp_sm1d_kernel<T, W><<<dim3((unsigned)p->nsub, p->nvec), block_threads(interp_sm1d_kernel<T, W>, p->threads),
                               smem, p->stream>>>(a);
  }
  return cudaGetLastError();
}

#define NUFFT_1D_CASES(FN)                                                               \
  switch (p->w) {                                                                        \
    case 2: return FN<T, 2>(p, c);   case 3: return FN<T, 3>(p, c);                      \
    case 4: return FN<T, 4>(p, c);   case 5: return FN<T, 5>(p, c);                      \
    case 6: return FN<T, 6>(p, c);   case 7: return FN<T, 7>(p, c);                      \
    case 8: return FN<T, 8>(p, c);   case 9: return FN<T, 9>(p, c);                      \
    case 10: return FN<T, 10>(p, c); case 11: return FN<T, 11>(p, c);                    \
    case 12: return FN<T, 12>(p, c); case 13: return FN<T, 13>(p, c);                    \
    case 14: return FN<T, 14>(p, c); case 15: return FN<T, 15>(p, c);                    \
    case 16: return FN<T, 16>(p, c);                                                     \
    default: return cudaErrorInvalidValue;                                               \
  }

template <typename T>
cudaError_t spread1d_t(const nufft_plan_s *p, const void *c) { NUFFT_1D_CASES(spread1d_w) }
template <typename T>
cudaError_t interp1d_t(const nufft_plan_s *p, void *c) { NUFFT_1D_CASES(interp1d_w) }

}  // namespace

cudaError_t launch_spread_1d(const nufft_plan_s *p, const void *c) {
  return p->dtype == 0 ? spread1d_t<float>(p, c) : spread1d_t<double>(p, c);
}

cudaError_t launch_interp_1d(const nufft_plan_s *p, void *c) {
  return p->dtype == 0 ? interp1d_t<float>(p, c) : interp1d_t<double>(p, c);
}

}  // namespace nufft
