// 3D single-precision interpolation (type 2 step 3, Sec. II-B c of the
// cuFINUFFT paper) over a staged padded bin, with the tile reads shared by
// points whose windows coincide.
//
// c_j = sum_l b_l psi(l h - x_j) reads the w^3 tile values of the window
// that starts at node l0(x_j) = ceil(g_j - w/2) in each dimension.  Points
// whose three window origins are equal read the same w^3 values: at the
// density of a sigma = 2 grid (about two points per fine cell) most points
// share their window with others.  A thread evaluates one group of at most K
// such points: each tile row is loaded once into registers and multiplied
// into the K points' row sums, so shared-memory reads per point fall to about
// half of one thread per point at K = 4, at the same multiply-adds per point.
//
// The groups are built once per setpts (group3d_build_kernel), one block per
// subproblem: the subproblem's sorted points are reordered by window origin
// (any order inside a subproblem is a valid sort), each origin's run is cut
// into groups of at most K, and one 32-bit record per group (first point
// inside the subproblem, size) is written next to the subproblem's points.
// Records are ordered by size, largest first, so warps that run K-point
// groups are not mixed with warps of single points; within one size they
// are dealt round robin over the window origin mod 16 (the bank pair a
// point's 8-byte tile reads start on), so the 16 lanes of a half warp
// mostly read distinct bank pairs.
//
// A point's sums are those of the thread-per-point kernel (the same weights,
// the same order of the multiply-adds), whichever group or slot it lands in.
#include "spreadinterp.cuh"

namespace nufft {
namespace {

constexpr int kBuildThreads = 256;
constexpr int kGroupThreads = 256;
constexpr int kRankBits = 13;  // ranks below 8192 (M_sub <= 8192)
constexpr int kMaxKeys = 1 << (31 - kRankBits);

__device__ __forceinline__ int g3_block_exclusive(int v, int *total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int before = warp == 0 ? 0 : warp_sums[warp - 1];
  *total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before + inc - v;
}

struct BuildArgs {
  Subproblem *sub;
  int32_t *perm;
  float *g1, *g2, *g3;
  uint32_t *grec;
  int m1, m2, m3;
};

// One block per subproblem.  Dynamic shared memory: R + 1 origin counters,
// then n (key, rank) words, then n staged points (x, y, z, caller index).
template <int W, int K>
__global__ void __launch_bounds__(kBuildThreads) group3d_build_kernel(BuildArgs a) {
  static_assert(K >= 1 && K <= 8, "group sizes fit the record");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int PAD = (W + 1) / 2;
  constexpr int S0 = PAD - W / 2;  // smallest window origin in the tile
  const int p1 = a.m1 + 2 * PAD, p2 = a.m2 + 2 * PAD;
  const int q1 = a.m1 + 1, q2 = a.m2 + 1;
  const int R = q1 * q2 * (a.m3 + 1);  // window origins minus S0 lie in [0, m_d]
  const Subproblem sp = a.sub[blockIdx.x];
  const int n = sp.count, base = sp.start;
  int *keyc = reinterpret_cast<int *>(smem_raw);
  int *pk = keyc + ((R + 1 + 3) & ~3);
  float4 *pts = reinterpret_cast<float4 *>(pk + ((n + 3) & ~3));
  __shared__ int cb[K * 16], cur[K * 16], cls_start[K + 1];
  const int tid = threadIdx.x, bd = blockDim.x;

  for (int i = tid; i <= R; i += bd) keyc[i] = 0;
  for (int i = tid; i < K * 16; i += bd) cb[i] = cur[i] = 0;
  __syncthreads();
  for (int k = tid; k < n; k += bd) {
    const float x = a.g1[base + k], y = a.g2[base + k], z = a.g3[base + k];
    const int r1 = min(max((int)es_ceil(x - 0.5f * W) + PAD - S0, 0), a.m1);
    const int r2 = min(max((int)es_ceil(y - 0.5f * W) + PAD - S0, 0), a.m2);
    const int r3 = min(max((int)es_ceil(z - 0.5f * W) + PAD - S0, 0), a.m3);
    const int key = (r3 * q2 + r2) * q1 + r1;
    pk[k] = key << kRankBits | atomicAdd(&keyc[key], 1);
    pts[k] = make_float4(x, y, z, __int_as_float(a.perm[base + k]));
  }
  __syncthreads();

  // bank pair of an origin's tile reads
  auto bucket_of = [&](int key) {
    const int r1 = key % q1, rr = key / q1;
    const int r2 = rr % q2, r3 = rr / q2;
    return (((r3 + S0) * p2 + r2 + S0) * p1 + r1 + S0) & 15;
  };
  // counts -> starts (in place); groups per (size class, bucket) on the way;
  // class c holds the groups of K - c points
  {
    const int per = (R + bd - 1) / bd;
    const int lo = min(tid * per, R), hi = min(lo + per, R);
    int sum = 0;
    for (int i = lo; i < hi; i++) {
      const int c = keyc[i];
      sum += c;
      if (c > 0) {
        const int b = bucket_of(i);
        const int full = c / K, rem = c - full * K;
        if (full) atomicAdd(&cb[b], full);
        if (rem) atomicAdd(&cb[(K - rem) * 16 + b], 1);
      }
    }
    int total;
    int ex = g3_block_exclusive(sum, &total);
    for (int i = lo; i < hi; i++) {
      const int c = keyc[i];
      keyc[i] = ex;
      ex += c;
    }
    if (tid == 0) keyc[R] = total;
  }
  __syncthreads();

  // points in origin order; class starts
  for (int k = tid; k < n; k += bd) {
    const int v = pk[k];
    const int pos = base + keyc[v >> kRankBits] + (v & ((1 << kRankBits) - 1));
    const float4 q = pts[k];
    a.g1[pos] = q.x;
    a.g2[pos] = q.y;
    a.g3[pos] = q.z;
    a.perm[pos] = __float_as_int(q.w);
  }
  if (tid == 0) {
    int acc = 0;
    for (int c = 0; c < K; c++) {
      cls_start[c] = acc;
      for (int b = 0; b < 16; b++) acc += cb[c * 16 + b];
    }
    cls_start[K] = acc;
    a.sub[blockIdx.x].groups = acc;
  }
  __syncthreads();

  // group records, round robin over the buckets within a class: the i-th
  // group of bucket b goes after every bucket's first i groups and after the
  // i-th groups of buckets b' < b
  auto place = [&](int c, int b, int rec) {
    const int i = atomicAdd(&cur[c * 16 + b], 1);
    int pos = cls_start[c];
#pragma unroll
    for (int b2 = 0; b2 < 16; b2++) {
      const int s = cb[c * 16 + b2];
      pos += min(s, i) + (b2 < b && s > i ? 1 : 0);
    }
    a.grec[base + pos] = (uint32_t)rec;
  };
  for (int key = tid; key < R; key += bd) {
    const int st = keyc[key], c = keyc[key + 1] - st;
    if (c == 0) continue;
    const int b = bucket_of(key);
    const int full = c / K, rem = c - full * K;
    for (int i = 0; i < full; i++) place(0, b, (st + i * K) | K << 16);
    if (rem) place(K - rem, b, (st + full * K) | rem << 16);
  }
}

// Interpolate the (at most Q) points of one group: sorted slots j0 .. j0 +
// size - 1, all with the same window origin; slots q >= size repeat j0 and
// are not written.
template <int W, int Q>
__device__ __forceinline__ void g3_group(const float2 *__restrict__ tile, int p1, int p2,
                                         const SIParams<float> &a, int j0, int size, uint64_t pol_stream,
                                         uint64_t pol_keep) {
  constexpr int PAD = (W + 1) / 2;
  constexpr int S0 = PAD - W / 2;
  const float scale = 2.0f / W;
  const float beta = a.beta;
  float kx[Q][W], ky[Q][W], dz[Q];
  int s1 = 0, s2 = 0, s3 = 0;
#pragma unroll
  for (int q = 0; q < Q; q++) {
    const int j = q < size ? j0 + q : j0;
    const float gx = ld_hint(a.g1 + j, pol_stream), gy = ld_hint(a.g2 + j, pol_stream),
                gz = ld_hint(a.g3 + j, pol_stream);
    const float lx = es_ceil(gx - 0.5f * W), ly = es_ceil(gy - 0.5f * W), lz = es_ceil(gz - 0.5f * W);
    if (q == 0) {  // window origin in the tile, in [S0, m + S0] for g in [0, m]
      s1 = min(max((int)lx + PAD, S0), a.m1 + S0);
      s2 = min(max((int)ly + PAD, S0), a.m2 + S0);
      s3 = min(max((int)lz + PAD, S0), a.m3 + S0);
    }
    const float dx = lx - gx, dy = ly - gy;
#pragma unroll
    for (int t = 0; t < W; t++) {
      kx[q][t] = es_fast((dx + float(t)) * scale, beta);
      ky[q][t] = es_fast((dy + float(t)) * scale, beta);
    }
    dz[q] = lz - gz;
  }
  float ar[Q], ai[Q];
#pragma unroll
  for (int q = 0; q < Q; q++) ar[q] = ai[q] = 0.0f;
#pragma unroll 1
  for (int i3 = 0; i3 < W; i3++) {
    float pr[Q], pi[Q];
#pragma unroll
    for (int q = 0; q < Q; q++) pr[q] = pi[q] = 0.0f;
#pragma unroll
    for (int i2 = 0; i2 < W; i2++) {
      const float2 *row = tile + ((s3 + i3) * p2 + s2 + i2) * p1 + s1;
      float2 b[W];
#pragma unroll
      for (int i1 = 0; i1 < W; i1++) b[i1] = row[i1];
#pragma unroll
      for (int q = 0; q < Q; q++) {
        float sr = 0.0f, si = 0.0f;
#pragma unroll
        for (int i1 = 0; i1 < W; i1++) {
          sr += b[i1].x * kx[q][i1];
          si += b[i1].y * kx[q][i1];
        }
        pr[q] += sr * ky[q][i2];
        pi[q] += si * ky[q][i2];
      }
    }
#pragma unroll
    for (int q = 0; q < Q; q++) {
      const float v3 = es_fast((dz[q] + float(i3)) * scale, beta);
      ar[q] += pr[q] * v3;
      ai[q] += pi[q] * v3;
    }
  }
#pragma unroll
  for (int q = 0; q < Q; q++)
    if (q < size) st_hint(a.c_out + ld_hint(a.perm + j0 + q, pol_stream), make_float2(ar[q], ai[q]), pol_keep);
}

template <int W, int K>
__global__ void __launch_bounds__(kGroupThreads, K <= 2 ? 3 : 2)
    interp_group3d_kernel(SIParams<float> a, const uint32_t *__restrict__ grec) {
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
  const uint64_t pol_stream = l2_evict_first(), pol_keep = l2_evict_last();
  const int tid = threadIdx.x, bd = blockDim.x;
  for (int base = tid; base < cells; base += 4 * bd) {
    C v[4];
    int at[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int t = base + u * bd;
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

  const int G = sp.groups;
  for (int base = 0; base < G; base += bd) {
    const int slot = base + tid;
    const uint32_t rec = slot < G ? ld_hint(reinterpret_cast<const int32_t *>(grec) + sp.start + slot,
                                           pol_stream)
                                  : 0u;
    const int j0 = sp.start + (int)(rec & 0xffffu), size = (int)(rec >> 16);
    const int qmax = __reduce_max_sync(0xffffffffu, size);
    if (K >= 4 && qmax >= 4) {
      g3_group<W, (K >= 4 ? K : 1)>(tile, p1, p2, a, j0, size, pol_stream, pol_keep);
    } else if (K >= 3 && qmax == 3) {
      g3_group<W, (K >= 3 ? 3 : 1)>(tile, p1, p2, a, j0, size, pol_stream, pol_keep);
    } else if (K >= 2 && qmax == 2) {
      g3_group<W, (K >= 2 ? 2 : 1)>(tile, p1, p2, a, j0, size, pol_stream, pol_keep);
    } else if (qmax == 1) {
      g3_group<W, 1>(tile, p1, p2, a, j0, size, pol_stream, pol_keep);
    }
  }
}

size_t build_smem(const nufft_plan_s *p) {
  const size_t R = (size_t)(p->m[0] + 1) * (p->m[1] + 1) * (p->m[2] + 1);
  const size_t n = (size_t)p->msub;
  return ((R + 1 + 3) & ~size_t(3)) * 4 + ((n + 3) & ~size_t(3)) * 4 + n * 16;
}

template <int W, int K>
cudaError_t build_wk(const nufft_plan_s *p) {
  BuildArgs a;
  a.sub = p->subprob;
  a.perm = p->perm;
  a.g1 = static_cast<float *>(p->gcoord[0]);
  a.g2 = static_cast<float *>(p->gcoord[1]);
  a.g3 = static_cast<float *>(p->gcoord[2]);
  a.grec = p->grec;
  a.m1 = p->m[0];
  a.m2 = p->m[1];
  a.m3 = p->m[2];
  const size_t smem = build_smem(p);
  cudaError_t e = allow_smem(group3d_build_kernel<W, K>, smem);
  if (e != cudaSuccess) return e;
  group3d_build_kernel<W, K><<<(unsigned)p->nsub, kBuildThreads, smem, p->stream>>>(a);
  return cudaGetLastError();
}

template <int W, int K>
cudaError_t interp_wk(const nufft_plan_s *p, void *c) {
  SIParams<float> a = make_params<float>(p);
  a.c_out = static_cast<float2 *>(c);
  const size_t smem = tile_cells(p) * sizeof(float2);
  cudaError_t e = allow_smem(interp_group3d_kernel<W, K>, smem);
  if (e != cudaSuccess) return e;
  interp_group3d_kernel<W, K><<<dim3((unsigned)p->nsub, p->nvec),
                                block_threads(interp_group3d_kernel<W, K>, p->threads), smem, p->stream>>>(
      a, p->grec);
  return cudaGetLastError();
}

template <int W>
cudaError_t build_w(const nufft_plan_s *p) {
  switch (p->igroup) {
    case 2: return build_wk<W, 2>(p);
    case 3: return build_wk<W, 3>(p);
    case 4: return build_wk<W, 4>(p);
    default: return cudaErrorInvalidValue;
  }
}

template <int W>
cudaError_t interp_w(const nufft_plan_s *p, void *c) {
  switch (p->igroup) {
    case 2: return interp_wk<W, 2>(p, c);
    case 3: return interp_wk<W, 3>(p, c);
    case 4: return interp_wk<W, 4>(p, c);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool group3d_supported(const nufft_plan_s *p, int smem_max) {
  if (p->dim != 3 || p->dtype != 0 || p->w < 2 || p->w > kGroup3DMaxWidth) return false;
  if (p->msub > (1 << kRankBits)) return false;
  const int64_t R = (int64_t)(p->m[0] + 1) * (p->m[1] + 1) * (p->m[2] + 1);
  if (R >= kMaxKeys) return false;
  return build_smem(p) <= (size_t)smem_max && tile_cells(p) * sizeof(float2) <= (size_t)smem_max;
}

cudaError_t build_groups3d(const nufft_plan_s *p) {
  if (p->nsub == 0) return cudaSuccess;
  switch (p->w) {
    case 2: return build_w<2>(p);
    case 3: return build_w<3>(p);
    case 4: return build_w<4>(p);
    case 5: return build_w<5>(p);
    case 6: return build_w<6>(p);
    case 7: return build_w<7>(p);
    case 8: return build_w<8>(p);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_interp_group3d(const nufft_plan_s *p, void *c) {
  switch (p->w) {
    case 2: return interp_w<2>(p, c);
    case 3: return interp_w<3>(p, c);
    case 4: return interp_w<4>(p, c);
    case 5: return interp_w<5>(p, c);
    case 6: return interp_w<6>(p, c);
    case 7: return interp_w<7>(p, c);
    case 8: return interp_w<8>(p, c);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nufft
