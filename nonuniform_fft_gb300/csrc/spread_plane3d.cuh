// Type 1 spreading in 3D with the subproblem's padded bin held in registers.
//
// Decomposition of the SM method of "cuFINUFFT: a load-balanced GPU library
// for general-purpose nonuniform FFTs" (Sec. III-A, Fig. 1, generalised to
// cuboid bins as that section describes): bin-sorted points, subproblems of at
// most M_sub points of one bin, accumulation of eq. (14) on a private padded
// bin (eq. (13)), periodic add-back into the fine grid (eq. (15)).  The padded
// bin lives in registers of one thread block:
//   * the bin is 32 - 2 ceil(w/2) cells wide in x: lane L of every warp owns
//     padded-bin column L;
//   * warp k owns the Z padded-bin planes kZ .. kZ+Z-1 (K warps, K Z planes);
//   * for each of its planes a lane keeps a window of w+1 padded-bin rows in
//     registers; the block walks the bin's rows in order and after each row
//     the lowest row of every window is complete: it is added to the fine
//     grid and the windows slide down one row.
// Setpts sorts a bin's points cell by cell (x fastest, then y, then z), so the
// points of bin row y in z-layer z form one contiguous run, and the points of
// that run whose x-window covers a lane's column form a contiguous sub-run.
// For every row the block stages, once per point, the kernel values of all
// the row's runs (w+1 "extended" values per dimension on the nodes
// cell - floor(w/2) .. cell - floor(w/2) + w, exactly w of them the support);
// each warp then visits the runs whose z-window reaches its planes, each lane
// the points whose x-window reaches its column.  No shared-memory atomics and
// no shared-memory read-modify-write.
#pragma once

#include <type_traits>

#include "df64.cuh"
#include "spread_regtile.cuh"

namespace nufft {

template <typename T, int W, int Z, int K, int STAGE_KB = 72>
struct Plane3D {
  static constexpr int PAD = (W + 1) / 2;
  static constexpr int HW = W / 2;
  static constexpr int WX = W + 1;
  static constexpr int VEC = 16 / (int)sizeof(T);
  // staged y weights: WX values, then the point's cell offset xb in slot WX
  // when the last 16-byte unit has room (else in an array of its own); rows
  // an odd number of 16-byte units apart (no bank conflicts between the 8
  // lanes of a quarter warp storing or loading 16 bytes each)
  static constexpr bool XB_IN_ROW = WX % VEC != 0;
  static constexpr int WXP = (WX + VEC - 1) / VEC * VEC;
  static constexpr int WYS = (WXP / VEC) % 2 == 0 ? WXP + VEC : WXP;
  static constexpr int WCS = WX | 1;        // odd row stride of the c * x-weight products
  // odd row stride of the z weights: the lanes of a warp read one column of
  // different points' rows, which an even stride folds onto a few banks
  static constexpr int WZS = WX | 1;
  static constexpr int M1 = 32 - 2 * PAD;   // bin width (x)
  static constexpr int P3 = K * Z;          // padded-bin planes
  static constexpr int M3 = P3 - 2 * PAD;   // bin depth (z)
  static constexpr int THREADS = 32 * K;
  // staged points per batch within STAGE_KB of dynamic shared memory (three
  // blocks of 8 warps share an SM); larger batches mean fewer block barriers
  static constexpr int PT_BYTES = (int)sizeof(T) * (WYS + WZS + 2 * WCS) + (XB_IN_ROW ? 0 : 4);
  static constexpr int S_FIT = (STAGE_KB * 1024 / PT_BYTES) / 32 * 32;
  static constexpr int S = S_FIT < 1024 ? S_FIT : 1024;
  static_assert(S >= 32, "staging buffer too small");
  static_assert(M1 >= 1 && M3 >= 1, "padded bin too small for this width");
};

template <typename T, int W, int Z, int K>
struct __align__(16) Plane3DStage {
  using G = Plane3D<T, W, Z, K>;
  typename Cplx<T>::type cwx[G::S][G::WCS];
  T wy[G::S][G::WYS];
  T wz[G::S][G::WZS];
  int xb[G::XB_IN_ROW ? 1 : G::S];
};

template <typename T>
struct Plane3DParams {
  using CT = typename Cplx<T>::type;
  const Subproblem *sub;
  const int32_t *perm;
  const T *g1, *g2, *g3;
  const int32_t *cell_starts;  // per (bin, cell), cells x fastest then y then z
  const CT *c_in;
  CT *grid;
  T beta_e;
  int n1, n2, n3;
  int m1, m2, m3;
  int nb1, nb2;
  int64_t cstride, gstride;  // per vector: M strengths, one fine grid
};

template <typename T, int W, int Z, int K>
__global__ void __launch_bounds__(Plane3D<T, W, Z, K>::THREADS)
    spread_plane3d_kernel(Plane3DParams<T> a) {
  using G = Plane3D<T, W, Z, K>;
  using CT = typename Cplx<T>::type;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_in += blockIdx.y * a.cstride;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Plane3DStage<T, W, Z, K> &stg = *reinterpret_cast<Plane3DStage<T, W, Z, K> *>(smem_raw);
  auto &s_wy = stg.wy;    // y weights; [WX]: cell offset xb
  auto &s_wz = stg.wz;
  auto &s_xbs = stg.xb;   // cell offsets, when not in s_wy
  auto &s_cwx = stg.cwx;  // c_j times the x weights
  // runs of the current row: one per z-layer of the subproblem
  __shared__ int r_lo[G::M3], r_hi[G::M3], r_pos[G::M3 + 1];
  __shared__ int r_cs[G::M3][G::M1 + 1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Subproblem sp = a.sub[blockIdx.x];
  const int b1 = sp.bin % a.nb1, rest = sp.bin / a.nb1;
  const int b2 = rest % a.nb2, b3 = rest / a.nb2;
  const int lo = sp.start, hi = sp.start + sp.count;
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int cpl = a.m1 * a.m2;  // cells per z-layer of a bin
  const int32_t *cs = a.cell_starts + (int64_t)sp.bin * cpl * a.m3;

  // z-layers spanned by this run of cell-sorted points (z is slowest)
  const int z_a = (int)floor(a.g3[lo]);
  const int z_b = (int)floor(a.g3[hi - 1]);
  const int nl = z_b - z_a + 1;

  // this warp's planes t = warp*Z + i are bin-relative z nodes t - PAD; a
  // point of z-layer zc reaches node t - PAD iff zc - HW <= t - PAD <= zc - HW + W
  const int t0 = warp * Z;
  // this lane's column x_rel = lane - PAD takes points of x-cells
  // [x_rel + HW - W, x_rel + HW]
  const int x_rel = lane - G::PAD;
  int xw_lo = x_rel + G::HW - W, xw_hi = x_rel + G::HW + 1;
  xw_lo = xw_lo < 0 ? 0 : xw_lo;
  xw_hi = xw_hi > a.m1 ? a.m1 : xw_hi;
  CT *col_base = a.grid + wrap_tile(b1 * a.m1 + x_rel, a.n1);
  int64_t plane_off[Z];
#pragma unroll
  for (int i = 0; i < Z; i++)
    plane_off[i] = (int64_t)wrap_tile(b3 * a.m3 - G::PAD + t0 + i, a.n3) * a.n2 * a.n1;
  const int row0 = b2 * a.m2 - G::PAD;  // fine-grid row of padded-bin row 0

  T acc_r[Z][G::WX], acc_i[Z][G::WX];
#pragma unroll
  for (int i = 0; i < Z; i++)
#pragma unroll
    for (int r = 0; r < G::WX; r++) acc_r[i][r] = acc_i[i][r] = T(0);

  for (int yc = 0; yc < a.m2; yc++) {
    // --- the row's runs (one per z-layer) and their cell starts -----------
    for (int e = tid; e < nl * (a.m1 + 1); e += G::THREADS) {
      const int l = e / (a.m1 + 1), x = e - l * (a.m1 + 1);
      r_cs[l][x] = cs[((z_a + l) * a.m2 + yc) * a.m1 + x];
    }
    __syncthreads();
    if (warp == 0) {
      int len = 0;
      if (lane < nl) {
        int s0 = r_cs[lane][0], s1 = r_cs[lane][a.m1];
        s0 = s0 > lo ? s0 : lo;
        s1 = s1 < hi ? s1 : hi;
        r_lo[lane] = s0;
        r_hi[lane] = s1 > s0 ? s1 : s0;
        len = s1 > s0 ? s1 - s0 : 0;
      }
      // inclusive scan of the run lengths over the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, len, o);
        if (lane >= o) len += u;
      }
      if (lane < nl) r_pos[lane + 1] = len;
      if (lane == 0) r_pos[0] = 0;
    }
    __syncthreads();
    const int total = r_pos[nl];

    for (int vs = 0; vs < total; vs += G::S) {
      const int ve = vs + G::S < total ? vs + G::S : total;
      // --- stage the batch: virtual positions vs .. ve-1 over the runs ----
      for (int v = vs + tid; v < ve; v += G::THREADS) {
        int l = 0;
        while (l + 1 < nl && r_pos[l + 1] <= v) l++;
        const int j = r_lo[l] + (v - r_pos[l]);
        const int q = v - vs;
        const int src = ld_hint(a.perm + j, pol_stream);
        const CT cv = ld_hint(a.c_in + src, pol_keep);
        T ex[G::WXP], ey[G::WXP], ez[G::WXP];
        const int xb = es_extended<T, W, G::WXP>(ld_hint(a.g1 + j, pol_stream), a.beta_e, ex);
        es_extended<T, W, G::WXP>(ld_hint(a.g2 + j, pol_stream), a.beta_e, ey);
        es_extended<T, W, G::WXP>(ld_hint(a.g3 + j, pol_stream), a.beta_e, ez);
        if constexpr (G::XB_IN_ROW)
          ey[G::WX < G::WXP ? G::WX : 0] = xb_pack<T>(xb);
        else
          s_xbs[q] = xb;
#pragma unroll
        for (int v = 0; v < G::WXP; v += G::VEC) Vec16<T>::put(&s_wy[q][v], &ey[v]);
#pragma unroll
        for (int s = 0; s < G::WX; s++) {
          s_wz[q][s] = ez[s];
          CT pr;
          pr.x = cv.x * ex[s];
          pr.y = cv.y * ex[s];
          s_cwx[q][s] = pr;
        }
      }
      __syncthreads();
      // --- visit: runs whose z-window reaches this warp's planes ----------
      for (int l = 0; l < nl; l++) {
        const int zc = z_a + l;
        // extended z-weight index of plane t0 + i for points of layer zc
        const int ez0 = (t0 - G::PAD) - (zc - G::HW);
        if (ez0 + Z - 1 < 0 || ez0 > W) continue;  // warp-uniform
        if (xw_lo >= xw_hi) continue;
        int j0 = r_cs[l][xw_lo], j1 = r_cs[l][xw_hi];
        j0 = j0 > r_lo[l] ? j0 : r_lo[l];
        j1 = j1 < r_hi[l] ? j1 : r_hi[l];
        // to batch slots
        int q0 = r_pos[l] + (j0 - r_lo[l]) - vs, q1 = r_pos[l] + (j1 - r_lo[l]) - vs;
        q0 = q0 > 0 ? q0 : 0;
        q1 = q1 < ve - vs ? q1 : ve - vs;
        for (int q = q0; q < q1; q++) {
          T wy[G::WXP];
#pragma unroll
          for (int v = 0; v < G::WXP; v += G::VEC) Vec16<T>::get(&s_wy[q][v], &wy[v]);
          int d;
          if constexpr (G::XB_IN_ROW)
            d = x_rel - xb_unpack(wy[G::WX < G::WXP ? G::WX : 0]);
          else
            d = x_rel - s_xbs[q];
          d = d < 0 ? 0 : (d > W ? W : d);
          const CT cw = s_cwx[q][d];
#pragma unroll
          for (int i = 0; i < Z; i++) {
            const int e = ez0 + i;
            const T wz = (e >= 0 && e <= W) ? s_wz[q][e < 0 ? 0 : (e > W ? W : e)] : T(0);
            const T cr = cw.x * wz, ci = cw.y * wz;
#pragma unroll
            for (int r = 0; r < G::WX; r++) {
              acc_r[i][r] += cr * wy[r];
              acc_i[i][r] += ci * wy[r];
            }
          }
        }
      }
      __syncthreads();
    }
    // --- padded-bin row yc - HW + PAD is complete in every plane ----------
    {
      const int64_t row_off = (int64_t)wrap_tile(row0 + yc - G::HW + G::PAD, a.n2) * a.n1;
#pragma unroll
      for (int i = 0; i < Z; i++)
        if (acc_r[i][0] != T(0) || acc_i[i][0] != T(0))
          grid_atomic_add(col_base + plane_off[i] + row_off, acc_r[i][0], acc_i[i][0]);
    }
#pragma unroll
    for (int i = 0; i < Z; i++) {
#pragma unroll
      for (int r = 0; r < W; r++) {
        acc_r[i][r] = acc_r[i][r + 1];
        acc_i[i][r] = acc_i[i][r + 1];
      }
      acc_r[i][W] = acc_i[i][W] = T(0);
    }
  }
  // the last w rows of every plane
#pragma unroll
  for (int r = 0; r < W; r++) {
    const int64_t row_off =
        (int64_t)wrap_tile(row0 + a.m2 - G::HW + G::PAD + r, a.n2) * a.n1;
#pragma unroll
    for (int i = 0; i < Z; i++)
      if (acc_r[i][r] != T(0) || acc_i[i][r] != T(0))
        grid_atomic_add(col_base + plane_off[i] + row_off, acc_r[i][r], acc_i[i][r]);
  }
}

// Double precision: the same register tile, with the multiply-accumulates in
// two-float arithmetic (df64.cuh).  Kernel values are evaluated in double
// per point and dimension, split once into two-floats at staging; the
// window accumulators are two-floats and are converted back to double when a
// row is added to the fine grid.
template <int W, int Z, int K, int STAGE_KB = 160>
struct Plane3DDF {
  static constexpr int PAD = (W + 1) / 2;
  static constexpr int HW = W / 2;
  static constexpr int WX = W + 1;
  static constexpr int M1 = 32 - 2 * PAD;
  static constexpr int P3 = K * Z;
  static constexpr int M3 = P3 - 2 * PAD;
  static constexpr int THREADS = 32 * K;
  static constexpr int WCS = WX | 1;  // odd stride of the 16-byte c * x-weight products
  // staged points per batch: the accumulators allow one block per SM, so the
  // staging buffer (dynamic shared memory) may take most of the SM's 228 KB;
  // fewer, larger batches mean fewer block barriers per bin row
  static constexpr int PT_BYTES = 8 * WX + 8 * WX + 16 * WCS + 4;
  static constexpr int S_FIT = (STAGE_KB * 1024 / PT_BYTES) / 32 * 32;
  static constexpr int S = S_FIT < 1024 ? S_FIT : 1024;
  static_assert(S >= 32, "staging buffer too small");
  static_assert(M1 >= 1 && M3 >= 1, "padded bin too small for this width");
};

struct DFC {  // complex two-float
  DF re, im;
};

template <int W, int Z, int K>
struct __align__(16) Plane3DDFStage {
  using G = Plane3DDF<W, Z, K>;
  DFC cwx[G::S][G::WCS];  // c_j times the x weights
  DF wy[G::S][G::WX];
  DF wz[G::S][G::WX];
  int xb[G::S];
};

template <int W, int Z, int K>
__global__ void __launch_bounds__(Plane3DDF<W, Z, K>::THREADS, 1)
    spread_plane3d_df_kernel(Plane3DParams<double> a) {
  using G = Plane3DDF<W, Z, K>;
  using CT = double2;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_in += blockIdx.y * a.cstride;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Plane3DDFStage<W, Z, K> &stg = *reinterpret_cast<Plane3DDFStage<W, Z, K> *>(smem_raw);
  auto &s_wy = stg.wy;
  auto &s_wz = stg.wz;
  auto &s_cwx = stg.cwx;
  auto &s_xb = stg.xb;
  __shared__ int r_lo[G::M3], r_hi[G::M3], r_pos[G::M3 + 1];
  __shared__ int r_cs[G::M3][G::M1 + 1];
  __shared__ DF s_exp2[64];
  fill_exp2_64(s_exp2);  // read after the first barrier below

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Subproblem sp = a.sub[blockIdx.x];
  const int b1 = sp.bin % a.nb1, rest = sp.bin / a.nb1;
  const int b2 = rest % a.nb2, b3 = rest / a.nb2;
  const int lo = sp.start, hi = sp.start + sp.count;
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int cpl = a.m1 * a.m2;
  const int32_t *cs = a.cell_starts + (int64_t)sp.bin * cpl * a.m3;
  const int z_a = (int)floor(a.g3[lo]);
  const int z_b = (int)floor(a.g3[hi - 1]);
  const int nl = z_b - z_a + 1;
  const int t0 = warp * Z;
  const int x_rel = lane - G::PAD;
  int xw_lo = x_rel + G::HW - W, xw_hi = x_rel + G::HW + 1;
  xw_lo = xw_lo < 0 ? 0 : xw_lo;
  xw_hi = xw_hi > a.m1 ? a.m1 : xw_hi;
  CT *col_base = a.grid + wrap_tile(b1 * a.m1 + x_rel, a.n1);
  int64_t plane_off[Z];
#pragma unroll
  for (int i = 0; i < Z; i++)
    plane_off[i] = (int64_t)wrap_tile(b3 * a.m3 - G::PAD + t0 + i, a.n3) * a.n2 * a.n1;
  const int row0 = b2 * a.m2 - G::PAD;

  DF acc_r[Z][G::WX], acc_i[Z][G::WX];
#pragma unroll
  for (int i = 0; i < Z; i++)
#pragma unroll
    for (int r = 0; r < G::WX; r++) acc_r[i][r] = acc_i[i][r] = DF{0.f, 0.f};

  for (int yc = 0; yc < a.m2; yc++) {
    for (int e = tid; e < nl * (a.m1 + 1); e += G::THREADS) {
      const int l = e / (a.m1 + 1), x = e - l * (a.m1 + 1);
      r_cs[l][x] = cs[((z_a + l) * a.m2 + yc) * a.m1 + x];
    }
    __syncthreads();
    if (warp == 0) {
      int len = 0;
      if (lane < nl) {
        int s0 = r_cs[lane][0], s1 = r_cs[lane][a.m1];
        s0 = s0 > lo ? s0 : lo;
        s1 = s1 < hi ? s1 : hi;
        r_lo[lane] = s0;
        r_hi[lane] = s1 > s0 ? s1 : s0;
        len = s1 > s0 ? s1 - s0 : 0;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, len, o);
        if (lane >= o) len += u;
      }
      if (lane < nl) r_pos[lane + 1] = len;
      if (lane == 0) r_pos[0] = 0;
    }
    __syncthreads();
    const int total = r_pos[nl];

    for (int vs = 0; vs < total; vs += G::S) {
      const int ve = vs + G::S < total ? vs + G::S : total;
      for (int v = vs + tid; v < ve; v += G::THREADS) {
        int l = 0;
        while (l + 1 < nl && r_pos[l + 1] <= v) l++;
        const int j = r_lo[l] + (v - r_pos[l]);
        const int q = v - vs;
        const int src = ld_hint(a.perm + j, pol_stream);
        const CT cv = ld_hint(a.c_in + src, pol_keep);
        const double gx = ld_hint(a.g1 + j, pol_stream), gy = ld_hint(a.g2 + j, pol_stream),
                     gz = ld_hint(a.g3 + j, pol_stream);
        // one dimension at a time, so only one array of kernel values is live
        // next to the accumulators; two-float kernel values and products
        // (native double here kept the FP64 pipe a quarter busy)
        const DF beta = df_from(a.beta_e);
        DF ek[G::WX];
        es_extended_df<W, G::WX>(gy, beta, ek, s_exp2);
#pragma unroll
        for (int t = 0; t < G::WX; t++) s_wy[q][t] = ek[t];
        es_extended_df<W, G::WX>(gz, beta, ek, s_exp2);
#pragma unroll
        for (int t = 0; t < G::WX; t++) s_wz[q][t] = ek[t];
        s_xb[q] = es_extended_df<W, G::WX>(gx, beta, ek, s_exp2);
        const DF cr = df_from(cv.x), ci = df_from(cv.y);
#pragma unroll
        for (int t = 0; t < G::WX; t++) {
          DFC pr;
          pr.re = df_mul(cr, ek[t]);
          pr.im = df_mul(ci, ek[t]);
          s_cwx[q][t] = pr;
        }
      }
      __syncthreads();
      for (int l = 0; l < nl; l++) {
        const int zc = z_a + l;
        const int ez0 = (t0 - G::PAD) - (zc - G::HW);
        if (ez0 + Z - 1 < 0 || ez0 > W) continue;  // warp-uniform
        if (xw_lo >= xw_hi) continue;
        int j0 = r_cs[l][xw_lo], j1 = r_cs[l][xw_hi];
        j0 = j0 > r_lo[l] ? j0 : r_lo[l];
        j1 = j1 < r_hi[l] ? j1 : r_hi[l];
        int q0 = r_pos[l] + (j0 - r_lo[l]) - vs, q1 = r_pos[l] + (j1 - r_lo[l]) - vs;
        q0 = q0 > 0 ? q0 : 0;
        q1 = q1 < ve - vs ? q1 : ve - vs;
        for (int q = q0; q < q1; q++) {
          int d = x_rel - s_xb[q];
          d = d < 0 ? 0 : (d > W ? W : d);
          const DFC cw = s_cwx[q][d];
#pragma unroll
          for (int i = 0; i < Z; i++) {
            const int e = ez0 + i;
            if (e < 0 || e > W) continue;
            const DF wz = s_wz[q][e];
            const DF pr = df_mul(cw.re, wz), pi = df_mul(cw.im, wz);
#pragma unroll
            for (int r = 0; r < G::WX; r++) {
              const DF wy = s_wy[q][r];
              df_fma(acc_r[i][r], pr, wy);
              df_fma(acc_i[i][r], pi, wy);
            }
          }
        }
      }
      __syncthreads();
    }
    {
      const int64_t row_off = (int64_t)wrap_tile(row0 + yc - G::HW + G::PAD, a.n2) * a.n1;
#pragma unroll
      for (int i = 0; i < Z; i++) {
        const double vr = df_to(acc_r[i][0]), vi = df_to(acc_i[i][0]);
        if (vr != 0.0 || vi != 0.0) grid_atomic_add(col_base + plane_off[i] + row_off, vr, vi);
      }
    }
#pragma unroll
    for (int i = 0; i < Z; i++) {
#pragma unroll
      for (int r = 0; r < W; r++) {
        acc_r[i][r] = acc_r[i][r + 1];
        acc_i[i][r] = acc_i[i][r + 1];
      }
      acc_r[i][W] = acc_i[i][W] = DF{0.f, 0.f};
    }
  }
#pragma unroll
  for (int r = 0; r < W; r++) {
    const int64_t row_off = (int64_t)wrap_tile(row0 + a.m2 - G::HW + G::PAD + r, a.n2) * a.n1;
#pragma unroll
    for (int i = 0; i < Z; i++) {
      const double vr = df_to(acc_r[i][r]), vi = df_to(acc_i[i][r]);
      if (vr != 0.0 || vi != 0.0) grid_atomic_add(col_base + plane_off[i] + row_off, vr, vi);
    }
  }
}

// Warps per block K and planes per warp Z for a width and precision: K Z
// padded planes, so the bin is K Z - 2 ceil(w/2) cells deep.  The register
// windows (2 Z (w+1) values per lane) must fit K warps in one SM.  Double
// precision at w >= 9 takes 10 warps (measured at w = 13: 113 ms against
// 119 ms for 8 warps of 3 planes and 151 ms for 16 warps of 2 planes).
template <typename T, int W>
struct Plane3DChoice {
  static constexpr bool F = sizeof(T) == 4;
  static constexpr int Z = 2;
  static constexpr int K = F ? (W <= 8 ? 8 : 16) : (W <= 8 ? 8 : 10);
};

template <typename T, int W>
cudaError_t spread_plane3d_w(const nufft_plan_s *p, const void *c) {
  using Ch = Plane3DChoice<T, W>;
  using G = Plane3D<T, W, Ch::Z, Ch::K>;
  Plane3DParams<T> a{};
  a.sub = p->subprob;
  a.perm = p->perm;
  a.g1 = static_cast<const T *>(p->gcoord[0]);
  a.g2 = static_cast<const T *>(p->gcoord[1]);
  a.g3 = static_cast<const T *>(p->gcoord[2]);
  a.cell_starts = p->cell_starts;
  a.c_in = static_cast<const typename Cplx<T>::type *>(c);
  a.grid = static_cast<typename Cplx<T>::type *>(p->grid);
  a.beta_e = (T)es_beta_e(p->beta, sizeof(T));
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
  if constexpr (std::is_same<T, double>::value) {
    const size_t smem = sizeof(Plane3DDFStage<W, Ch::Z, Ch::K>);
    const cudaError_t e = allow_smem(spread_plane3d_df_kernel<W, Ch::Z, Ch::K>, smem);
    if (e != cudaSuccess) return e;
    spread_plane3d_df_kernel<W, Ch::Z, Ch::K>
        <<<dim3((unsigned)p->nsub, p->nvec), Plane3DDF<W, Ch::Z, Ch::K>::THREADS, smem, p->stream>>>(a);
  } else {
    const size_t smem = sizeof(Plane3DStage<T, W, Ch::Z, Ch::K>);
    const cudaError_t e = allow_smem(spread_plane3d_kernel<T, W, Ch::Z, Ch::K>, smem);
    if (e != cudaSuccess) return e;
    spread_plane3d_kernel<T, W, Ch::Z, Ch::K><<<dim3((unsigned)p->nsub, p->nvec), G::THREADS, smem, p->stream>>>(a);
  }
  return cudaGetLastError();
}

// Bin size the kernel is built for: 32 - 2 ceil(w/2) by m2 by K Z - 2 ceil(w/2).
template <typename T>
void plane3d_bins_t(int w, int *m1, int *m3) {
  const int pad = (w + 1) / 2;
  const bool f = sizeof(T) == 4;
  const int z = 2, k = f ? (w <= 8 ? 8 : 16) : (w <= 8 ? 8 : 10);
  *m1 = 32 - 2 * pad;
  *m3 = k * z - 2 * pad;
}

template <typename T>
cudaError_t launch_spread_plane3d(const nufft_plan_s *p, const void *c) {
  switch (p->w) {
    case 2: return spread_plane3d_w<T, 2>(p, c);
    case 3: return spread_plane3d_w<T, 3>(p, c);
    case 4: return spread_plane3d_w<T, 4>(p, c);
    case 5: return spread_plane3d_w<T, 5>(p, c);
    case 6: return spread_plane3d_w<T, 6>(p, c);
    case 7: return spread_plane3d_w<T, 7>(p, c);
    case 8: return spread_plane3d_w<T, 8>(p, c);
    case 9: return spread_plane3d_w<T, 9>(p, c);
    case 10: return spread_plane3d_w<T, 10>(p, c);
    case 11: return spread_plane3d_w<T, 11>(p, c);
    case 12: return spread_plane3d_w<T, 12>(p, c);
    case 13: return spread_plane3d_w<T, 13>(p, c);
    case 14: return spread_plane3d_w<T, 14>(p, c);
    case 15: return spread_plane3d_w<T, 15>(p, c);
    case 16: return spread_plane3d_w<T, 16>(p, c);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nufft
