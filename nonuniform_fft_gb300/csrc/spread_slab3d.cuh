// Type 1 spreading in 3D, single precision, with bins one fine-grid cell
// thick in z ("slab" bins) and the whole padded bin of one column in the
// registers of one lane.
//
// Decomposition of the SM method of "cuFINUFFT: a load-balanced GPU library
// for general-purpose nonuniform FFTs" (Sec. III-A, Fig. 1, cuboid bins):
// bin-sorted points, subproblems of at most M_sub points of one bin,
// accumulation of eq. (14) on a private padded bin (eq. (13)), periodic
// add-back into the fine grid (eq. (15)).  Here a bin is m1 x m2 x 1 cells
// and one warp takes a subproblem:
//   * lane L owns padded-bin column L (the bin is 32 - 2 ceil(w/2) cells
//     wide), for all w+1 z-planes a point of the slab can reach;
//   * the warp walks the bin's rows in order; each lane keeps, per plane, a
//     window of w+1 padded-bin rows in registers ((w+1)^2 complex values)
//     and adds c_j phi_x phi_y phi_z of its run of the row's points;
//   * after a row the lowest row of every plane's window is complete: it is
//     added to the fine grid, and the windows slide down one row.
// A point costs w+1 lane-visits, each loading its y and z weights and one
// product c_j phi_x from the warp's staging buffer and doing (w+1)^2
// complex multiply-adds, with no block-wide barrier anywhere.  The price is
// the z padding: every row flush adds w+1 planes for one layer of points.
// Setpts sorts a bin's points cell by cell (x fastest, then y), so the
// points of one row whose x-window covers a lane form a contiguous run.
#pragma once

#include "spread_regtile.cuh"

namespace nufft {

template <int W>
struct Slab3D {
  static constexpr int PAD = (W + 1) / 2;   // ceil(w/2), eq. (13)
  static constexpr int HW = W / 2;          // floor(w/2)
  static constexpr int WX = W + 1;          // extended window
  static constexpr int WXP = (WX + 3) / 4 * 4;
  // 16-byte rows of the y weights (the cell offset in a spare slot when there
  // is one) and of the z weights, an odd number of 16-byte units apart
  static constexpr bool XB_IN_ROW = WX % 4 != 0;
  static constexpr int ROWS16 = (WXP / 4) % 2 == 0 ? WXP + 4 : WXP;
  static constexpr int WCS = WX | 1;        // odd row stride of the c * x-weight products
  static constexpr int M1 = 32 - 2 * PAD;   // bin width (x)
  static constexpr int S = 64;              // staged points per batch
  static constexpr int WARPS = 4;
  // blocks per SM the registers are sized for: 3 up to w = 7 (at w = 7 the
  // cap of 168 registers spills 20 bytes and takes the 3D bench spread from
  // 4.87 to 4.38 ms; 4 blocks, 128 registers, spill far more: 9.8 ms)
  static constexpr int MIN_BLOCKS = W <= 7 ? 3 : 2;
};

template <int W>
struct __align__(16) Slab3DStage {
  using G = Slab3D<W>;
  float wy[G::S][G::ROWS16];   // y weights; [WX]: cell offset xb when it fits
  float wz[G::S][G::ROWS16];   // z weights
  float2 cwx[G::S][G::WCS];    // c_j times the x weights
  int xb[G::XB_IN_ROW ? 1 : G::S];
};

struct Slab3DParams {
  const Subproblem *sub;
  int nsub;
  const int32_t *perm;
  const float *g1, *g2, *g3;
  const int32_t *cell_starts;  // per (bin, cell): first sorted slot; cells x fastest, then y
  const float2 *c_in;
  float2 *grid;
  float beta_e;
  int n1, n2, n3;
  int m1, m2;
  int nb1, nb2;
  int64_t cstride, gstride;  // per vector: M strengths, one fine grid
};

template <int W>
__global__ void __launch_bounds__(32 * Slab3D<W>::WARPS, Slab3D<W>::MIN_BLOCKS)
    spread_slab3d_kernel(Slab3DParams a) {
  using G = Slab3D<W>;
  a.grid += blockIdx.y * a.gstride;  // vector blockIdx.y of a batched launch
  a.c_in += blockIdx.y * a.cstride;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Slab3DStage<W> &st = reinterpret_cast<Slab3DStage<W> *>(smem_raw)[warp];
  const int sidx = blockIdx.x * G::WARPS + warp;
  if (sidx >= a.nsub) return;  // whole warp leaves together
  const Subproblem sp = a.sub[sidx];
  const int b1 = sp.bin % a.nb1, rest = sp.bin / a.nb1;
  const int b2 = rest % a.nb2, b3 = rest / a.nb2;  // b3: the bin's z cell
  const int lo = sp.start, hi = sp.start + sp.count;
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int32_t *cs = a.cell_starts + (int64_t)sp.bin * (a.m1 * a.m2);

  // rows of the bin that this run of cell-sorted points spans
  const int y_first = (int)floorf(a.g2[lo]);
  const int y_last = (int)floorf(a.g2[hi - 1]);

  // lane's column x_rel = lane - PAD takes points of x-cells [x_rel + HW - W, x_rel + HW]
  const int x0 = lane - G::PAD;
  int xw_lo = x0 + G::HW - W, xw_hi = x0 + G::HW + 1;
  xw_lo = xw_lo < 0 ? 0 : xw_lo;
  xw_hi = xw_hi > a.m1 ? a.m1 : xw_hi;
  const int col = wrap_tile(b1 * a.m1 + x0, a.n1);
  const int row0 = b2 * a.m2 - G::PAD;  // fine-grid row of tile row 0 (before wrapping)
  const int64_t plane_cells = (int64_t)a.n1 * a.n2;

  // acc[p][r]: plane p (z node b3 - HW + p), window slot r (tile row yc - HW + PAD + r)
  float acc_r[G::WX][G::WX], acc_i[G::WX][G::WX];
#pragma unroll
  for (int p = 0; p < G::WX; p++)
#pragma unroll
    for (int r = 0; r < G::WX; r++) acc_r[p][r] = acc_i[p][r] = 0.f;

  auto flush_row = [&](int tile_row, int slot) {
    const int64_t roff = (int64_t)wrap_tile(row0 + tile_row, a.n2) * a.n1 + col;
#pragma unroll
    for (int p = 0; p < G::WX; p++) {
      if (acc_r[p][slot] != 0.f || acc_i[p][slot] != 0.f)
        grid_atomic_add(a.grid + (int64_t)wrap_tile(b3 - G::HW + p, a.n3) * plane_cells + roff,
                        acc_r[p][slot], acc_i[p][slot]);
    }
  };

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
      float gx[PER], gy[PER], gz[PER];
#pragma unroll
      for (int u = 0; u < PER; u++) {
        const int q = lane + 32 * u;
        src[u] = 0;
        gx[u] = gy[u] = gz[u] = 0.f;
        if (q < nb) {
          src[u] = ld_hint(a.perm + bs + q, pol_stream);
          gx[u] = ld_hint(a.g1 + bs + q, pol_stream);
          gy[u] = ld_hint(a.g2 + bs + q, pol_stream);
          gz[u] = ld_hint(a.g3 + bs + q, pol_stream);
        }
      }
      float2 cv[PER];
#pragma unroll
      for (int u = 0; u < PER; u++)
        if (lane + 32 * u < nb) cv[u] = ld_hint(a.c_in + src[u], pol_keep);
#pragma unroll
      for (int u = 0; u < PER; u++) {
        const int q = lane + 32 * u;
        if (q < nb) {
          float ex[G::WXP], ey[G::WXP], ez[G::WXP];
          const int xb = es_extended<float, W, G::WXP>(gx[u], a.beta_e, ex);
          es_extended<float, W, G::WXP>(gy[u], a.beta_e, ey);
          es_extended<float, W, G::WXP>(gz[u], a.beta_e, ez);  // the slab's one cell: planes 0..W
          if constexpr (G::XB_IN_ROW)
            ey[G::WX] = xb_pack<float>(xb);
          else
            st.xb[q] = xb;
#pragma unroll
          for (int v = 0; v < G::WXP; v += 4) {
            Vec16<float>::put(&st.wy[q][v], &ey[v]);
            Vec16<float>::put(&st.wz[q][v], &ez[v]);
          }
#pragma unroll
          for (int e = 0; e < G::WX; e++) st.cwx[q][e] = make_float2(cv[u].x * ex[e], cv[u].y * ex[e]);
        }
      }
      __syncwarp();
      const int j0 = llo > bs ? llo : bs, j1 = lhi < bs + nb ? lhi : bs + nb;
      for (int j = j0; j < j1; j++) {
        const int q = j - bs;
        float wy[G::WXP], wz[G::WXP];
#pragma unroll
        for (int v = 0; v < G::WXP; v += 4) {
          Vec16<float>::get(&st.wy[q][v], &wy[v]);
          Vec16<float>::get(&st.wz[q][v], &wz[v]);
        }
        int xbq;
        if constexpr (G::XB_IN_ROW)
          xbq = xb_unpack(wy[G::WX < G::WXP ? G::WX : 0]);
        else
          xbq = st.xb[q];
        // index of this lane's product in the point's row: in [0, W] for
        // points of the lane's window
        int e0 = x0 - xbq;
        e0 = e0 < 0 ? 0 : (e0 > W ? W : e0);
        const float2 cw = st.cwx[q][e0];
#pragma unroll
        for (int p = 0; p < G::WX; p++) {
          const float cr = cw.x * wz[p], ci = cw.y * wz[p];
#pragma unroll
          for (int r = 0; r < G::WX; r++) {
            acc_r[p][r] += cr * wy[r];
            acc_i[p][r] += ci * wy[r];
          }
        }
      }
      __syncwarp();
    }
    // tile row yc - HW + PAD is complete in every plane: add it to the fine
    // grid (eq. (15)), then slide the windows down one row
    flush_row(yc - G::HW + G::PAD, 0);
#pragma unroll
    for (int p = 0; p < G::WX; p++) {
#pragma unroll
      for (int r = 0; r < W; r++) {
        acc_r[p][r] = acc_r[p][r + 1];
        acc_i[p][r] = acc_i[p][r + 1];
      }
      acc_r[p][W] = acc_i[p][W] = 0.f;
    }
  }
  // the last w tile rows of every plane
#pragma unroll
  for (int r = 0; r < W; r++) flush_row(y_last + 1 - G::HW + G::PAD + r, r);
}

template <int W>
cudaError_t spread_slab3d_w(const nufft_plan_s *p, const void *c) {
  using G = Slab3D<W>;
  Slab3DParams a{};
  a.sub = p->subprob;
  a.nsub = (int)p->nsub;
  a.perm = p->perm;
  a.g1 = static_cast<const float *>(p->gcoord[0]);
  a.g2 = static_cast<const float *>(p->gcoord[1]);
  a.g3 = static_cast<const float *>(p->gcoord[2]);
  a.cell_starts = p->cell_starts;
  a.c_in = static_cast<const float2 *>(c);
  a.grid = static_cast<float2 *>(p->grid);
  a.beta_e = (float)es_beta_e(p->beta, sizeof(float));
  a.n1 = (int)p->n[0];
  a.n2 = (int)p->n[1];
  a.n3 = (int)p->n[2];
  a.m1 = p->m[0];
  a.m2 = p->m[1];
  a.nb1 = p->nb[0];
  a.nb2 = p->nb[1];
  a.cstride = p->M;
  a.gstride = grid_cells(p);
  const unsigned blocks = (unsigned)((p->nsub + G::WARPS - 1) / G::WARPS);
  const size_t smem = G::WARPS * sizeof(Slab3DStage<W>);
  cudaError_t e = allow_smem(spread_slab3d_kernel<W>, smem);
  if (e != cudaSuccess) return e;
  spread_slab3d_kernel<W><<<dim3(blocks, p->nvec), 32 * G::WARPS, smem, p->stream>>>(a);
  return cudaGetLastError();
}

}  // namespace nufft
