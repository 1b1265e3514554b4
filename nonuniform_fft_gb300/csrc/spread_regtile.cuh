// Type 1 spreading with the subproblem's padded bin held in registers
// ("register tile"), 2D.
//
// Same decomposition as the SM method of "cuFINUFFT: a load-balanced GPU
// library for general-purpose nonuniform FFTs" (Sec. III-A, Fig. 1): points
// are bin-sorted, each bin's points are cut into subproblems of at most M_sub
// points, a subproblem accumulates eq. (14) on a private copy of its padded
// bin (p_i = m_i + 2 ceil(w/2), eq. (13)) and adds it back into the fine grid
// with periodic wrapping (eq. (15)).  What differs is where the padded bin
// lives and who accumulates into it:
//   * one warp per subproblem; the bin is 32 C - 2 ceil(w/2) cells wide, so
//     the padded bin has 32 C columns and lane L owns columns L C .. L C + C - 1
//     (C = 4 for complex64, 2 for complex128);
//   * setpts sorts the points of a bin cell by cell (x fastest), so the points
//     of one fine-grid row whose x-window covers a lane's columns form one
//     contiguous run, found from the cell starts;
//   * the warp walks the subproblem's rows in order; each lane walks its own
//     run of points of the row and adds c_j phi_x phi_y into a window of w+1
//     registers (the w+1 tile rows the row's points can reach);
//   * once a row is done, the lowest tile row of the window can receive
//     nothing more: it is added to the fine grid and the window slides down
//     one row.  No shared-memory atomics, no shared-memory read-modify-write,
//     and 2 C (w+1) accumulator registers per lane whatever the bin height.
// Per point and dimension the w kernel values are computed once, into a
// per-warp staging buffer, as w+1 "extended" values on the nodes
// cell - floor(w/2) .. cell - floor(w/2) + w: exactly w of them are the
// point's support (l0 = ceil(g - w/2), z in [-1, 1)), the other is zero.
#pragma once

#include "spreadinterp.cuh"

namespace nufft {

template <typename T, int W, int C>
struct RowSlide2D {
  static constexpr int PAD = (W + 1) / 2;   // ceil(w/2), eq. (13)
  static constexpr int HW = W / 2;          // floor(w/2)
  static constexpr int WX = W + 1;          // extended window
  static constexpr int VEC = 16 / (int)sizeof(T);
  // staged y weights: WX values, then the point's cell offset xb in slot WX
  // when the last 16-byte unit has room for it (else in an array of its own,
  // rather than a whole extra unit per lane-visit)
  static constexpr bool XB_IN_ROW = WX % VEC != 0;
  static constexpr int WXP = (WX + VEC - 1) / VEC * VEC;
  // row stride of the y weights: an odd number of 16-byte units, so that the
  // 8 lanes of a quarter warp moving 16 bytes each hit 8 different bank quads
  static constexpr int WYS = (WXP / VEC) % 2 == 0 ? WXP + VEC : WXP;
  static constexpr int WXE = W + 2 * C - 1;  // x weights seen by C columns, zero-padded
  static constexpr int WCS = WXE | 1;        // odd row stride of the c * x-weight products
  static constexpr int M1 = 32 * C - 2 * PAD;  // bin width: C tile columns per lane
  // staged points per batch (measured on the 2D bench workload: 64 beats 96
  // for one column per lane although 96 holds a whole bin row; the wider
  // rows of two columns per lane prefer 96)
  static constexpr int S = sizeof(T) == 4 ? (C == 2 && W <= 7 ? 96 : 64) : 32;
  static constexpr int WARPS = 4;
};

// 16-byte vector of T.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  using type = float4;
  static __device__ __forceinline__ void put(float *dst, const float *v) {
    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
  }
  static __device__ __forceinline__ void get(const float *src, float *v) {
    const float4 t = *reinterpret_cast<const float4 *>(src);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  }
};
template <> struct Vec16<double> {
  using type = double2;
  static __device__ __forceinline__ void put(double *dst, const double *v) {
    *reinterpret_cast<double2 *>(dst) = make_double2(v[0], v[1]);
  }
  static __device__ __forceinline__ void get(const double *src, double *v) {
    const double2 t = *reinterpret_cast<const double2 *>(src);
    v[0] = t.x; v[1] = t.y;
  }
};

// Per-warp staging buffer of one batch of points.
template <typename T, int W, int C>
struct __align__(16) RegStage {
  using G = RowSlide2D<T, W, C>;
  T wy[G::S][G::WYS];                          // y weights; [WX]: cell offset xb
  typename Cplx<T>::type cwx[G::S][G::WCS];    // c_j times the x weights
  int xb[G::XB_IN_ROW ? 1 : G::S];             // cell offsets, when not in wy
};

// es_extended in two-float arithmetic (double-precision plans).
template <int W, int WX>
__device__ __forceinline__ int es_extended_df(double g, DF beta, DF (&ext)[WX], const DF *exp2_64) {
  constexpr int HW = W / 2;
  const double cellf = floor(g);
  DF k[W];
  const int l0 = es_weights_df<W>(g, beta, k, exp2_64);
  const int shift = l0 - ((int)cellf - HW);  // 0 or 1
#pragma unroll
  for (int s = 0; s < WX; s++) {
    const DF v0 = s < W ? k[s < W ? s : 0] : DF{0.f, 0.f};
    const DF v1 = (s >= 1 && s <= W) ? k[s >= 1 && s <= W ? s - 1 : 0] : DF{0.f, 0.f};
    ext[s] = shift ? v1 : v0;
  }
  return (int)cellf - HW;
}

// The cell offset xb travels in a spare slot of the staged y weights: as
// the int's bits in single precision (no conversion on either side), as an
// exactly representable value in double.
template <typename T>
__device__ __forceinline__ T xb_pack(int v);
template <>
__device__ __forceinline__ float xb_pack<float>(int v) { return __int_as_float(v); }
template <>
__device__ __forceinline__ double xb_pack<double>(int v) { return (double)v; }
__device__ __forceinline__ int xb_unpack(float v) { return __float_as_int(v); }
__device__ __forceinline__ int xb_unpack(double v) { return (int)v; }

template <typename T>
struct RegParams {
  using CT = typename Cplx<T>::type;
  const Subproblem *sub;
  int nsub;
  const int32_t *perm;
  const T *g1, *g2;
  const int32_t *cell_starts;  // per (bin, cell): first sorted slot; bin-major, x fastest
  const CT *c_in;
  CT *grid;
  T beta_e;
  int n1, n2;
  int m1, m2;  // runtime bin size (<= M1, M2 on tiny grids)
  int nb1;
  int64_t cstride, gstride;  // per vector: M strengths, one fine grid
};

// Extended kernel values of one coordinate g (bin-relative, in [cell, cell+1)):
// ext[s] = phi on node (cell - HW + s) if that node is in the support, else 0.
template <typename T, int W, int WXP>
__device__ __forceinline__ int es_extended(T g, T beta_e, T (&ext)[WXP]) {
  constexpr int HW = W / 2;
  const T cellf = floor(g);
  const T l0 = ceil(g - T(0.5) * T(W));
  const int shift = (int)(l0 - (cellf - T(HW)));  // 0 or 1
  const T d = l0 - g;
  const T scale = T(2) / T(W);
  T k[W];
#pragma unroll
  for (int t = 0; t < W; t++) k[t] = es_fast((d + T(t)) * scale, beta_e);
#pragma unroll
  for (int s = 0; s < WXP; s++) {
    T v0 = s < W ? k[s < W ? s : 0] : T(0);
    T v1 = (s >= 1 && s <= W) ? k[s >= 1 && s <= W ? s - 1 : 0] : T(0);
    ext[s] = shift ? v1 : v0;
  }
  return (int)cellf - HW;
}

template <typename T, int W, int C>
__global__ void __launch_bounds__(128) spread_regtile2d_kernel(RegParams<T> a) {
  using G = RowSlide2D<T, W, C>;
  using CT = typename Cplx<T>::type;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_in += blockIdx.y * a.cstride;
  using Stage = RegStage<T, W, C>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Stage &st = reinterpret_cast<Stage *>(smem_raw)[warp];
  const int sidx = blockIdx.x * G::WARPS + warp;
  if (sidx >= a.nsub) return;  // whole warp leaves together
  const Subproblem sp = a.sub[sidx];
  const int b1 = sp.bin % a.nb1, b2 = sp.bin / a.nb1;
  const int lo = sp.start, hi = sp.start + sp.count;
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int32_t *cs = a.cell_starts + (int64_t)sp.bin * (a.m1 * a.m2);

  // rows of the bin that this run of cell-sorted points spans
  const int y_first = (int)floor(a.g2[lo]);
  const int y_last = (int)floor(a.g2[hi - 1]);

  // this lane's tile columns x_rel = lane*C + cc - PAD take points whose cell
  // x_c has x_rel - (x_c - HW) in [0, W] for some cc
  const int x0 = lane * C - G::PAD;  // x_rel of the lane's first column
  int xw_lo = x0 + G::HW - W;
  int xw_hi = x0 + C + G::HW;  // exclusive
  xw_lo = xw_lo < 0 ? 0 : xw_lo;
  xw_hi = xw_hi > a.m1 ? a.m1 : xw_hi;
  int col[C];
#pragma unroll
  for (int cc = 0; cc < C; cc++) col[cc] = wrap_tile(b1 * a.m1 + x0 + cc, a.n1);
  const int row0 = b2 * a.m2 - G::PAD;  // fine-grid row of tile row 0 (before wrapping)

  // window slot r holds tile row (yc - HW + PAD + r) of this lane's columns
  T acc_r[C][G::WX], acc_i[C][G::WX];
#pragma unroll
  for (int cc = 0; cc < C; cc++)
#pragma unroll
    for (int r = 0; r < G::WX; r++) acc_r[cc][r] = acc_i[cc][r] = T(0);

  for (int yc = y_first; yc <= y_last; yc++) {
    const int32_t *row = cs + yc * a.m1;
    const int r0 = row[0], r1 = row[a.m1];
    const int rlo = r0 > lo ? r0 : lo, rhi = r1 < hi ? r1 : hi;
    int llo = rhi, lhi = rhi;
    if (xw_lo < xw_hi) {
      llo = row[xw_lo];
      lhi = row[xw_hi];
      llo = llo > rlo ? llo : rlo;
      lhi = lhi < rhi ? lhi : rhi;
    }
    for (int bs = rlo; bs < rhi; bs += G::S) {
      const int nb = (bs + G::S < rhi ? bs + G::S : rhi) - bs;
      // stage the batch: all loads first, then kernel values and stores
      constexpr int PER = G::S / 32;
      int src[PER];
      T gx[PER], gy[PER];
#pragma unroll
      for (int u = 0; u < PER; u++) {
        const int q = lane + 32 * u;
        src[u] = 0;
        gx[u] = gy[u] = T(0);
        if (q < nb) {
          src[u] = ld_hint(a.perm + bs + q, pol_stream);
          gx[u] = ld_hint(a.g1 + bs + q, pol_stream);
          gy[u] = ld_hint(a.g2 + bs + q, pol_stream);
        }
      }
      CT cv[PER];
#pragma unroll
      for (int u = 0; u < PER; u++)
        if (lane + 32 * u < nb) cv[u] = ld_hint(a.c_in + src[u], pol_keep);
#pragma unroll
      for (int u = 0; u < PER; u++) {
        const int q = lane + 32 * u;
        if (q < nb) {
          T ex[G::WXP], ey[G::WXP];
          const int xb = es_extended<T, W, G::WXP>(gx[u], a.beta_e, ex);
          es_extended<T, W, G::WXP>(gy[u], a.beta_e, ey);
          if constexpr (G::XB_IN_ROW)
            ey[G::WX] = xb_pack<T>(xb);
          else
            st.xb[q] = xb;
#pragma unroll
          for (int v = 0; v < G::WXP; v += G::VEC) Vec16<T>::put(&st.wy[q][v], &ey[v]);
#pragma unroll
          for (int e = 0; e < G::WXE; e++) {
            const int s = e - (C - 1);
            const T wxe = (s >= 0 && s <= W) ? ex[s >= 0 && s <= W ? s : 0] : T(0);
            CT v;
            v.x = cv[u].x * wxe;
            v.y = cv[u].y * wxe;
            st.cwx[q][e] = v;
          }
        }
      }
      __syncwarp();
      const int j0 = llo > bs ? llo : bs, j1 = lhi < bs + nb ? lhi : bs + nb;
      for (int j = j0; j < j1; j++) {
        const int q = j - bs;
        T wy[G::WXP];
#pragma unroll
        for (int v = 0; v < G::WXP; v += G::VEC) Vec16<T>::get(&st.wy[q][v], &wy[v]);
        // index of column cc's product in the zero-padded row: in
        // [0, W + 2C - 2] for points of this lane's window
        int xbq;
        if constexpr (G::XB_IN_ROW)
          xbq = xb_unpack(wy[G::WX < G::WXP ? G::WX : 0]);
        else
          xbq = st.xb[q];
        int e0 = x0 - xbq + (C - 1);
        e0 = e0 < 0 ? 0 : (e0 > W + C - 1 ? W + C - 1 : e0);
#pragma unroll
        for (int cc = 0; cc < C; cc++) {
          const CT cw = st.cwx[q][e0 + cc];
          const T cr = cw.x, ci = cw.y;
#pragma unroll
          for (int r = 0; r < G::WX; r++) {
            acc_r[cc][r] += cr * wy[r];
            acc_i[cc][r] += ci * wy[r];
          }
        }
      }
      __syncwarp();
    }
    // tile row yc - HW + PAD is complete: add it to the fine grid (eq. (15)),
    // then slide the window down one row
    {
      CT *grow_ = a.grid + (int64_t)wrap_tile(row0 + yc - G::HW + G::PAD, a.n2) * a.n1;
#pragma unroll
      for (int cc = 0; cc < C; cc++)
        if (acc_r[cc][0] != T(0) || acc_i[cc][0] != T(0))
          grid_atomic_add(grow_ + col[cc], acc_r[cc][0], acc_i[cc][0]);
    }
#pragma unroll
    for (int cc = 0; cc < C; cc++) {
#pragma unroll
      for (int r = 0; r < W; r++) {
        acc_r[cc][r] = acc_r[cc][r + 1];
        acc_i[cc][r] = acc_i[cc][r + 1];
      }
      acc_r[cc][W] = acc_i[cc][W] = T(0);
    }
  }
  // the last w tile rows
#pragma unroll
  for (int r = 0; r < W; r++) {
    CT *grow_ = a.grid + (int64_t)wrap_tile(row0 + y_last + 1 - G::HW + G::PAD + r, a.n2) * a.n1;
#pragma unroll
    for (int cc = 0; cc < C; cc++)
      if (acc_r[cc][r] != T(0) || acc_i[cc][r] != T(0))
        grid_atomic_add(grow_ + col[cc], acc_r[cc][r], acc_i[cc][r]);
  }
}

template <typename T, int W, int C>
cudaError_t spread_regtile2d_wc(const nufft_plan_s *p, const void *c) {
  using G = RowSlide2D<T, W, C>;
  RegParams<T> a{};
  a.sub = p->subprob;
  a.nsub = (int)p->nsub;
  a.perm = p->perm;
  a.g1 = static_cast<const T *>(p->gcoord[0]);
  a.g2 = static_cast<const T *>(p->gcoord[1]);
  a.cell_starts = p->cell_starts;
  a.c_in = static_cast<const typename Cplx<T>::type *>(c);
  a.grid = static_cast<typename Cplx<T>::type *>(p->grid);
  a.beta_e = (T)es_beta_e(p->beta, sizeof(T));
  a.n1 = (int)p->n[0];
  a.n2 = (int)p->n[1];
  a.m1 = p->m[0];
  a.m2 = p->m[1];
  a.nb1 = p->nb[0];
  a.cstride = p->M;
  a.gstride = grid_cells(p);
  const unsigned blocks = (unsigned)((p->nsub + G::WARPS - 1) / G::WARPS);
  const size_t smem = G::WARPS * sizeof(RegStage<T, W, C>);
  cudaError_t e = allow_smem(spread_regtile2d_kernel<T, W, C>, smem);
  if (e != cudaSuccess) return e;
  spread_regtile2d_kernel<T, W, C><<<dim3(blocks, p->nvec), 32 * G::WARPS, smem, p->stream>>>(a);
  return cudaGetLastError();
}

// Columns per lane as resolved at setpts (p->regtile_cols; p->m[0] was set
// by regtile2d_bins for the same choice).
template <typename T, int W>
cudaError_t spread_regtile2d_w(const nufft_plan_s *p, const void *c) {
  switch (p->regtile_cols) {
    case 1: return spread_regtile2d_wc<T, W, 1>(p, c);
    case 2: return spread_regtile2d_wc<T, W, 2>(p, c);
    case 4: return spread_regtile2d_wc<T, W, 4>(p, c);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_spread_regtile2d(const nufft_plan_s *p, const void *c) {
  switch (p->w) {
    case 2: return spread_regtile2d_w<T, 2>(p, c);
    case 3: return spread_regtile2d_w<T, 3>(p, c);
    case 4: return spread_regtile2d_w<T, 4>(p, c);
    case 5: return spread_regtile2d_w<T, 5>(p, c);
    case 6: return spread_regtile2d_w<T, 6>(p, c);
    case 7: return spread_regtile2d_w<T, 7>(p, c);
    case 8: return spread_regtile2d_w<T, 8>(p, c);
    case 9: return spread_regtile2d_w<T, 9>(p, c);
    case 10: return spread_regtile2d_w<T, 10>(p, c);
    case 11: return spread_regtile2d_w<T, 11>(p, c);
    case 12: return spread_regtile2d_w<T, 12>(p, c);
    case 13: return spread_regtile2d_w<T, 13>(p, c);
    case 14: return spread_regtile2d_w<T, 14>(p, c);
    case 15: return spread_regtile2d_w<T, 15>(p, c);
    case 16: return spread_regtile2d_w<T, 16>(p, c);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nufft
