// Type 1 spreading in 3D, single precision, with bins one window origin
// thick in z ("slab" bins) and the whole padded bin of one column in the
// registers of one lane.
//
// Decomposition of the SM method of "cuFINUFFT: a load-balanced GPU library
// for general-purpose nonuniform FFTs" (Sec. III-A, Fig. 1, cuboid bins):
// bin-sorted points, subproblems of at most M_sub points of one bin,
// accumulation of eq. (14) on a private padded bin (eq. (13)), periodic
// add-back into the fine grid (eq. (15)).  Setpts bins these plans' points
// by window origin rather than by cell: a point belongs to the bin of q =
// l0 + floor(w/2), l0 = ceil(g - w/2) the first of its w nodes, so its
// window is nodes q - floor(w/2) .. q - floor(w/2) + w - 1 and the padded
// bin needs only w - 1 columns of padding.  A bin is m1 x m2 x 1 origins and
// one warp takes a subproblem:
//   * lane L owns padded-bin column L (bin x origin L - floor(w/2); the bin
//     is 33 - w origins wide), for the w z-planes of the slab's points;
//   * the warp walks the bin's origin rows in order; each lane keeps, per
//     plane, a window of w padded-bin rows in registers (w^2 complex values)
//     and adds c_j phi_x phi_y phi_z of its run of the row's points;
//   * after a row the lowest row of every plane's window is complete: it is
//     added to the fine grid, and the windows slide down one row.
// A point costs w lane-visits, each loading its y and z weights and one
// product c_j phi_x from the warp's staging buffer and doing w^2 complex
// multiply-adds, with no block-wide barrier anywhere.  (Binned by cell, a
// point's window could start at either of two nodes in each dimension, and
// each lane-visit did (w+1)^2 multiply-adds for w+1 lanes: 4.37 against
// 3.40 ms on the 3D single-precision workload.)  Setpts sorts a bin's points
// origin by origin (x fastest, then y), so the points of one row whose
// x-window covers a lane form a contiguous run.
#pragma once

#include "spread_regtile.cuh"

namespace nufft {

template <int W>
struct Slab3D {
  static constexpr int HW = W / 2;          // left padding floor(w/2)
  static constexpr int WP = (W + 3) / 4 * 4;
  // 16-byte rows of the y weights (the x origin in a spare slot when there
  // is one) and of the z weights, an odd number of 16-byte units apart
  static constexpr bool XQ_IN_ROW = W % 4 != 0;
  static constexpr int ROWS16 = (WP / 4) % 2 == 0 ? WP + 4 : WP;
  static constexpr int WCS = W | 1;         // odd row stride of the c * x-weight products
  static constexpr int M1 = 33 - W;         // bin width (x origins)
  static constexpr int S = 64;              // staged points per batch
  static constexpr int WARPS = 4;
  // blocks per SM the registers are sized for: 3 up to w = 7, 2 above (at
  // w = 8 the 64 complex accumulators alone take 128 registers)
  static constexpr int MIN_BLOCKS = W <= 7 ? 3 : 2;
};

template <int W>
struct __align__(16) Slab3DStage {
  using G = Slab3D<W>;
  float wy[G::S][G::ROWS16];   // y weights; [W]: x origin when it fits
  float wz[G::S][G::ROWS16];   // z weights
  float2 cwx[G::S][G::WCS];    // c_j times the x weights
  int xq[G::XQ_IN_ROW ? 1 : G::S];
};

struct Slab3DParams {
  const Subproblem *sub;
  int nsub;
  const int32_t *perm;
  const float *g1, *g2, *g3;
  const int32_t *cell_starts;  // per (bin, origin): first sorted slot; x fastest, then y
  const float2 *c_in;
  float2 *grid;
  float beta_e;
  int n1, n2, n3;
  int m1, m2;
  int nb1, nb2;
  int64_t cstride, gstride;  // per vector: M strengths, one fine grid
};

// Window origin of a bin-relative coordinate, shifted by floor(w/2): the
// bin-relative origin setpts binned the point by, ceil(g - oc) with oc = 1/2
// for odd w and 0 for even w (exact in float: setpts keeps g within (q - 1
// + oc, q + oc] of its origin q).
template <int W>
__device__ __forceinline__ int slab_origin(float g) {
  return (int)ceilf(g - (W % 2 ? 0.5f : 0.0f));
}

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
  const int b2 = rest % a.nb2, b3 = rest / a.nb2;  // b3: the slab's z origin
  const int lo = sp.start, hi = sp.start + sp.count;
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int32_t *cs = a.cell_starts + (int64_t)sp.bin * (a.m1 * a.m2);

  // origin rows of the bin that this run of sorted points spans
  const int y_first = slab_origin<W>(a.g2[lo]);
  const int y_last = slab_origin<W>(a.g2[hi - 1]);

  // lane's column (bin x origin L - floor(w/2)) takes the points of x origins [L - W + 1, L]
  int xw_lo = lane - W + 1, xw_hi = lane + 1;
  xw_lo = xw_lo < 0 ? 0 : xw_lo;
  xw_hi = xw_hi > a.m1 ? a.m1 : xw_hi;
  const int col = wrap_tile(b1 * a.m1 - G::HW + lane, a.n1);
  const int row0 = b2 * a.m2 - G::HW;  // fine-grid row of padded row 0 (before wrapping)
  const int64_t plane_cells = (int64_t)a.n1 * a.n2;

  // acc[p][r]: plane p (z node b3 - HW + p), window slot r (padded row yq + r)
  float acc_r[W][W], acc_i[W][W];
#pragma unroll
  for (int p = 0; p < W; p++)
#pragma unroll
    for (int r = 0; r < W; r++) acc_r[p][r] = acc_i[p][r] = 0.f;

  auto flush_row = [&](int prow, int slot) {
    const int64_t roff = (int64_t)wrap_tile(row0 + prow, a.n2) * a.n1 + col;
#pragma unroll
    for (int p = 0; p < W; p++) {
      if (acc_r[p][slot] != 0.f || acc_i[p][slot] != 0.f)
        grid_atomic_add(a.grid + (int64_t)wrap_tile(b3 - G::HW + p, a.n3) * plane_cells + roff,
                        acc_r[p][slot], acc_i[p][slot]);
    }
  };

  for (int yq = y_first; yq <= y_last; yq++) {
    const int32_t *row = cs + yq * a.m1;
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
          // windows at the point's x origin, the row's y origin and the
          // slab's z origin (0): nodes origin - floor(w/2) + t
          float kx[W], ky[G::WP], kz[G::WP];
          const int xq = slab_origin<W>(gx[u]);
          es_weights_at<float, W>(gx[u], xq - G::HW, a.beta_e, kx);
          es_weights_at<float, W>(gy[u], yq - G::HW, a.beta_e, reinterpret_cast<float(&)[W]>(ky));
          es_weights_at<float, W>(gz[u], -G::HW, a.beta_e, reinterpret_cast<float(&)[W]>(kz));
#pragma unroll
          for (int v = W; v < G::WP; v++) ky[v] = kz[v] = 0.f;
          if constexpr (G::XQ_IN_ROW)
            ky[W] = xb_pack<float>(xq);
          else
            st.xq[q] = xq;
#pragma unroll
          for (int v = 0; v < G::WP; v += 4) {
            Vec16<float>::put(&st.wy[q][v], &ky[v]);
            Vec16<float>::put(&st.wz[q][v], &kz[v]);
          }
#pragma unroll
          for (int e = 0; e < W; e++) st.cwx[q][e] = make_float2(cv[u].x * kx[e], cv[u].y * kx[e]);
        }
      }
      __syncwarp();
      const int j0 = llo > bs ? llo : bs, j1 = lhi < bs + nb ? lhi : bs + nb;
      for (int j = j0; j < j1; j++) {
        const int q = j - bs;
        float wy[G::WP], wz[G::WP];
#pragma unroll
        for (int v = 0; v < G::WP; v += 4) {
          Vec16<float>::get(&st.wy[q][v], &wy[v]);
          Vec16<float>::get(&st.wz[q][v], &wz[v]);
        }
        int xq;
        if constexpr (G::XQ_IN_ROW)
          xq = xb_unpack(wy[G::XQ_IN_ROW ? W : 0]);
        else
          xq = st.xq[q];
        // index of this lane's product in the point's row: in [0, W) for
        // points of the lane's run
        int e0 = lane - xq;
        e0 = e0 < 0 ? 0 : (e0 > W - 1 ? W - 1 : e0);
        const float2 cw = st.cwx[q][e0];
#pragma unroll
        for (int p = 0; p < W; p++) {
          const float cr = cw.x * wz[p], ci = cw.y * wz[p];
#pragma unroll
          for (int r = 0; r < W; r++) {
            acc_r[p][r] += cr * wy[r];
            acc_i[p][r] += ci * wy[r];
          }
        }
      }
      __syncwarp();
    }
    // padded row yq is complete in every plane: add it to the fine grid
    // (eq. (15)), then slide the windows down one row
    flush_row(yq, 0);
#pragma unroll
    for (int p = 0; p < W; p++) {
#pragma unroll
      for (int r = 0; r < W - 1; r++) {
        acc_r[p][r] = acc_r[p][r + 1];
        acc_i[p][r] = acc_i[p][r + 1];
      }
      acc_r[p][W - 1] = acc_i[p][W - 1] = 0.f;
    }
  }
  // the last w - 1 padded rows of every plane
#pragma unroll
  for (int r = 0; r < W - 1; r++) flush_row(y_last + 1 + r, r);
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
