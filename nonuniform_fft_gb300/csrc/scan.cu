// Exclusive prefix sum of int32 counts (the scan step of the bin sort in
// Sec. III-A of the cuFINUFFT paper: bin counts -> bin starts, and
// subproblems per bin -> first subproblem of each bin).
//
// Three launches, no inter-block waiting: (1) every block reduces its tile,
// (2) one block scans the tile sums, (3) every block scans its tile again and
// adds its offset.  Inside a block the scan is built from warp shuffles.
#include "nufft_internal.cuh"

namespace nufft {
namespace {

constexpr int kThreads = 1024;
constexpr int kPerThread = 4;
constexpr int kTile = kThreads * kPerThread;

__device__ __forceinline__ int warp_inclusive(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// Exclusive scan of one value per thread across the block; returns the
// thread's exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive(int v, int *total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = warp_inclusive(v);
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
    s = warp_inclusive(s);
    warp_sums[lane] = s;
  }
  __syncthreads();
  int before = warp == 0 ? 0 : warp_sums[warp - 1];
  *total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before + inc - v;
}

__global__ void __launch_bounds__(kThreads) tile_sums(const int32_t *in, int64_t n, int32_t *sums) {
  const int64_t base = (int64_t)blockIdx.x * kTile + (int64_t)threadIdx.x * kPerThread;
  int s = 0;
#pragma unroll
  for (int i = 0; i < kPerThread; i++)
    if (base + i < n) s += in[base + i];
  int total;
  block_exclusive(s, &total);
  if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

// One block: exclusive scan of the tile sums in place (chunks of kTile with
// a running carry); writes the grand total to sums[nt].
__global__ void __launch_bounds__(kThreads) scan_sums(int32_t *sums, int64_t nt) {
  int carry = 0;
  for (int64_t off = 0; off < nt; off += kTile) {
    const int64_t base = off + (int64_t)threadIdx.x * kPerThread;
    int v[kPerThread];
    int s = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; i++) {
      v[i] = base + i < nt ? sums[base + i] : 0;
      s += v[i];
    }
    int total;
    int ex = block_exclusive(s, &total) + carry;
#pragma unroll
    for (int i = 0; i < kPerThread; i++) {
      if (base + i < nt) sums[base + i] = ex;
      ex += v[i];
    }
    carry += total;
  }
  if (threadIdx.x == 0) sums[nt] = carry;
}

__global__ void __launch_bounds__(kThreads) scan_tiles(const int32_t *in, int32_t *out, int64_t n,
                                                       const int32_t *sums, int64_t nt) {
  const int64_t base = (int64_t)blockIdx.x * kTile + (int64_t)threadIdx.x * kPerThread;
  int v[kPerThread];
  int s = 0;
#pragma unroll
  for (int i = 0; i < kPerThread; i++) {
    v[i] = base + i < n ? in[base + i] : 0;
    s += v[i];
  }
  int total;
  int ex = block_exclusive(s, &total) + sums[blockIdx.x];
#pragma unroll
  for (int i = 0; i < kPerThread; i++) {
    if (base + i < n) out[base + i] = ex;
    ex += v[i];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) out[n] = sums[nt];
}

}  // namespace

int64_t scan_scratch_len(int64_t n) { return (n + kTile - 1) / kTile + 1; }

cudaError_t exclusive_scan(const int32_t *in, int32_t *out, int64_t n, int32_t *scratch,
                           cudaStream_t s) {
  if (n <= 0) {
    return cudaMemsetAsync(out, 0, sizeof(int32_t), s);
  }
  const int64_t nt = (n + kTile - 1) / kTile;
  tile_sums<<<(unsigned)nt, kThreads, 0, s>>>(in, n, scratch);
  scan_sums<<<1, kThreads, 0, s>>>(scratch, nt);
  scan_tiles<<<(unsigned)nt, kThreads, 0, s>>>(in, out, n, scratch, nt);
  return cudaGetLastError();
}

}  // namespace nufft
