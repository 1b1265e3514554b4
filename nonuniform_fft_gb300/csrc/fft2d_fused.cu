// Fine-grid FFT of 2D single-precision plans, pruned to the modes that the
// correction step keeps and fused with that step.
//
// Source: "cuFINUFFT: a load-balanced GPU library for general-purpose
// nonuniform FFTs", Sec. II.  Type 1 step 2 (eq. (9)) transforms the whole
// n1 x n2 fine grid and step 3 (eq. (10)) keeps only the modes k in I_N,
// scaled by p1(k1) p2(k2).  Here the 2D FFT is taken as a pass along x (one
// length-n1 transform per fine-grid row) and a pass along y:
//   * x pass: of each row's n1 frequencies only the N1 of the kept k1 are
//     written, transposed into a workspace T[i1][y] (N1 x n2);
//   * y pass: each row of T is transformed, the N2 kept frequencies are
//     scaled by p1 p2 and written to f, so the correction costs no pass of
//     its own.
// Type 2 (eq. (11), (12)) runs the same in reverse: the y pass reads f,
// applies p1 p2 and the zero padding on the fly and writes T; the x pass
// pads each T column's N1 entries to n1 and writes the whole fine grid.
// Against a full 2D FFT plus a correction kernel this skips half of the
// second pass and reads and writes the padding region of the fine grid once
// instead of several times.
//
// Each transform is a radix-8 Stockham FFT (the last radix 4 or 2) of
// L = 2^a complex values, 128 <= L <= 4096, in shared memory.  Stage s with
// stride Ns (product of the earlier radices) takes, for butterfly j, the R
// values at j + r L/R, multiplies value r by w^{(j mod Ns) r L/(Ns R)}
// (w = exp(s 2 pi i / L), s the plan's sign), takes their R-point DFT and
// stores value r at (j div Ns) Ns R + (j mod Ns) + r Ns; after the last stage
// the data are in natural order.  A block owns KV consecutive vectors (rows
// of the fine grid or of T; KV = 4 up to L = 1024, else 2, so that a block
// has at most 512 threads and two fit an SM): the KV threads that handle the
// same index of the KV vectors sit in adjacent lanes, so the accesses across
// vectors are runs of 8 KV bytes.  Shared index i lives at i + floor(i/16),
// with the vectors 16/KV (mod 16) elements apart: every stage's 8-byte loads
// and stores then take the minimum 2 wavefronts per warp.
#include <algorithm>
#include <cmath>
#include <vector>

#include "nufft_internal.cuh"

namespace nufft {
namespace {

constexpr int kMinLog = 7;        // L = 128
constexpr int kMaxLog = 12;       // L = 4096

__host__ __device__ constexpr int padded(int i) { return i + (i >> 4); }

template <int L>
struct Shape {
  static constexpr int TPV = L / 8 < 256 ? L / 8 : 256;   // threads per vector
  static constexpr int KV = L / 8 <= 128 ? 4 : 2;          // vectors per block
  static constexpr int THREADS = KV * TPV;
  static constexpr int LP0 = padded(L - 1) + 1;
  static constexpr int LP = LP0 + ((16 / KV - LP0 % 16) + 16) % 16;  // == 16/KV (mod 16)
  static constexpr size_t SMEM = (size_t)KV * LP * sizeof(float2);
  // three blocks per SM (at most 42 registers) where one radix-8 butterfly
  // per thread and stage leaves room for it
  static constexpr int MIN_BLOCKS = L <= 2048 ? 3 : 1;
};

__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
  return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}
// s i z
template <int S>
__device__ __forceinline__ float2 mul_si(float2 z) {
  return S > 0 ? make_float2(-z.y, z.x) : make_float2(z.y, -z.x);
}

// R-point DFTs X_k = sum_m x_m exp(s 2 pi i m k / R), in place, natural order.
template <int S>
__device__ __forceinline__ void dft4(float2 &x0, float2 &x1, float2 &x2, float2 &x3) {
  const float2 a0 = cadd(x0, x2), a1 = csub(x0, x2);
  const float2 b0 = cadd(x1, x3), b1 = mul_si<S>(csub(x1, x3));
  x0 = cadd(a0, b0);
  x2 = csub(a0, b0);
  x1 = cadd(a1, b1);
  x3 = csub(a1, b1);
}

template <int R, int S>
struct Dft;

template <int S>
struct Dft<2, S> {
  static __device__ __forceinline__ void run(float2 (&x)[2]) {
    const float2 t = x[0];
    x[0] = cadd(t, x[1]);
    x[1] = csub(t, x[1]);
  }
};

template <int S>
struct Dft<4, S> {
  static __device__ __forceinline__ void run(float2 (&x)[4]) { dft4<S>(x[0], x[1], x[2], x[3]); }
};

// 8 = 2 x 4: the DFTs of the even and the odd samples, combined with the
// factors exp(s 2 pi i k / 8), k = 0..3.
template <int S>
struct Dft<8, S> {
  static __device__ __forceinline__ void run(float2 (&x)[8]) {
    float2 a0 = x[0], a1 = x[2], a2 = x[4], a3 = x[6];
    float2 b0 = x[1], b1 = x[3], b2 = x[5], b3 = x[7];
    dft4<S>(a0, a1, a2, a3);
    dft4<S>(b0, b1, b2, b3);
    const float h = 0.70710678118654752f;
    b1 = make_float2(h * (b1.x - S * b1.y), h * (S * b1.x + b1.y));    // (1 + s i) / sqrt 2
    b2 = mul_si<S>(b2);                                                 // s i
    b3 = make_float2(-h * (b3.x + S * b3.y), h * (S * b3.x - b3.y));   // (-1 + s i) / sqrt 2
    x[0] = cadd(a0, b0);
    x[4] = csub(a0, b0);
    x[1] = cadd(a1, b1);
    x[5] = csub(a1, b1);
    x[2] = cadd(a2, b2);
    x[6] = csub(a2, b2);
    x[3] = cadd(a3, b3);
    x[7] = csub(a3, b3);
  }
};

// Radix of the stage with stride NS: 8 while at least 8 remain, else the rest.
template <int L, int NS>
struct StageRadix {
  static constexpr int R = L / NS >= 8 ? 8 : L / NS;
};

// Stages with stride NS > 1 up to the last, on one vector's shared buffer.
// tw holds exp(s 2 pi i t / Lt) for t < Lt, read at stride Lt / L.  The last
// stage hands (frequency index, value) to out instead of storing.
template <int L, int S, int NS, class Out>
__device__ __forceinline__ void fft_stages(float2 *buf, const float2 *__restrict__ tw, int tw_step, int jt,
                                           Out &out) {
  constexpr int R = StageRadix<L, NS>::R;
  constexpr int TPV = Shape<L>::TPV;
  constexpr int G = (L / R) / TPV;  // butterflies per thread
  constexpr bool LAST = NS * R == L;
  float2 x[G][R];
#pragma unroll
  for (int g = 0; g < G; g++) {
    const int j = jt + g * TPV;
#pragma unroll
    for (int r = 0; r < R; r++) x[g][r] = buf[padded(j + r * (L / R))];
  }
  if constexpr (!LAST) __syncthreads();  // in place: every load before any store
#pragma unroll
  for (int g = 0; g < G; g++) {
    const int j = jt + g * TPV;
    const int k = j & (NS - 1);
    {
      // u^r, u = w^{k L/(NS R)}, for r < R from one table read:
      // u^{2m} = (u^m)^2 and u^{2m+1} = u^{m+1} u^m, at most three complex
      // products deep (r = 5, 6, 7)
      float2 wr[R];
      wr[1 % R] = __ldg(tw + (int64_t)(k * (L / (NS * R))) * tw_step);
#pragma unroll
      for (int r = 2; r < R; r++)
        wr[r] = (r % 2 == 0) ? cmul(wr[r / 2], wr[r / 2]) : cmul(wr[r / 2 + 1], wr[r / 2]);
#pragma unroll
      for (int r = 1; r < R; r++) x[g][r] = cmul(x[g][r], wr[r]);
    }
    Dft<R, S>::run(x[g]);
    const int base = (j / NS) * NS * R + k;
#pragma unroll
    for (int r = 0; r < R; r++) {
      if constexpr (LAST)
        out(base + r * NS, x[g][r]);
      else
        buf[padded(base + r * NS)] = x[g][r];
    }
  }
  if constexpr (!LAST) {
    __syncthreads();
    fft_stages<L, S, NS * R>(buf, tw, tw_step, jt, out);
  }
}

// Whole transform of one vector: the first stage (stride 1, no twiddles)
// takes its inputs from in(q) straight from global memory.  Every thread of
// the block must call it (it synchronises the block).
template <int L, int S, class In, class Out>
__device__ __forceinline__ void fft_vector(float2 *buf, const float2 *__restrict__ tw, int tw_step, int jt,
                                           In &in, Out &out) {
  constexpr int TPV = Shape<L>::TPV;
  constexpr int G = (L / 8) / TPV;
  float2 x[G][8];
#pragma unroll
  for (int g = 0; g < G; g++) {
    const int j = jt + g * TPV;
#pragma unroll
    for (int r = 0; r < 8; r++) x[g][r] = in(j + r * (L / 8));
  }
#pragma unroll
  for (int g = 0; g < G; g++) {
    const int j = jt + g * TPV;
    Dft<8, S>::run(x[g]);
#pragma unroll
    for (int r = 0; r < 8; r++) buf[padded(8 * j + r)] = x[g][r];
  }
  __syncthreads();
  fft_stages<L, S, 8>(buf, tw, tw_step, jt, out);
}

struct FusedArgs {
  const float2 *in;       // the pass's source
  float2 *out;            // the pass's destination
  float2 *grid;           // type 1 x pass: the fine grids it reads and then clears
  const float *p1, *p2;   // correction factors, N1 and N2 entries (increasing k)
  const float2 *tw;       // exp(s 2 pi i t / tw_len), t < tw_len
  int tw_len;
  int n1, n2, N1, N2;
  int h1, h2;             // floor(N_i / 2): mode k has index k + h_i
  int64_t in_stride, out_stride;  // per vector of a batched launch
};

// mode index of fine-grid frequency q (length-n axis), or -1 when q holds no
// mode of I_N (eq. (10): mode k sits at k mod n)
__device__ __forceinline__ int mode_of(int q, int N, int h, int n) {
  if (q < N - h) return q + h;
  if (q >= n - h) return q - n + h;
  return -1;
}

// type 1, x pass: KV fine-grid rows -> T[i1][y]; afterwards each thread
// clears the grid cells it read, so the next type 1 execute finds the fine
// grid zeroed (the clear of step 1 folded into this pass)
template <int L, int S>
__global__ void __launch_bounds__(Shape<L>::THREADS, Shape<L>::MIN_BLOCKS) fft_t1_rows_kernel(FusedArgs a) {
  extern __shared__ __align__(16) float2 fft_smem[];
  constexpr int KV = Shape<L>::KV;
  const int v = threadIdx.x % KV, jt = threadIdx.x / KV;
  const int y = blockIdx.x * KV + v;
  float2 *row = a.grid + blockIdx.y * a.in_stride + (int64_t)y * L;
  float2 *T = a.out + blockIdx.y * a.out_stride;
  auto in = [&](int q) { return row[q]; };
  auto out = [&](int q, float2 val) {
    const int i1 = mode_of(q, a.N1, a.h1, L);
    if (i1 >= 0) T[(int64_t)i1 * a.n2 + y] = val;
  };
  fft_vector<L, S>(fft_smem + v * Shape<L>::LP, a.tw, a.tw_len / L, jt, in, out);
  // the same cells as the first stage's loads (one thread each)
  constexpr int TPV = Shape<L>::TPV;
#pragma unroll
  for (int g = 0; g < (L / 8) / TPV; g++)
#pragma unroll
    for (int r = 0; r < 8; r++) row[jt + g * TPV + r * (L / 8)] = make_float2(0.f, 0.f);
}

// type 1, y pass + correction: KV rows i1 of T -> f[i2][i1] p1(i1) p2(i2)
template <int L, int S>
__global__ void __launch_bounds__(Shape<L>::THREADS, Shape<L>::MIN_BLOCKS) fft_t1_cols_kernel(FusedArgs a) {
  extern __shared__ __align__(16) float2 fft_smem[];
  constexpr int KV = Shape<L>::KV;
  const int v = threadIdx.x % KV, jt = threadIdx.x / KV;
  const int i1 = blockIdx.x * KV + v;
  const bool ok = i1 < a.N1;
  const float2 *trow = a.in + blockIdx.y * a.in_stride + (int64_t)(ok ? i1 : 0) * L;
  float2 *f = a.out + blockIdx.y * a.out_stride;
  const float s1 = ok ? a.p1[i1] : 0.f;
  auto in = [&](int q) { return ok ? trow[q] : make_float2(0.f, 0.f); };
  auto out = [&](int q, float2 val) {
    const int i2 = mode_of(q, a.N2, a.h2, L);
    if (ok && i2 >= 0) {
      const float s = s1 * a.p2[i2];
      f[(int64_t)i2 * a.N1 + i1] = make_float2(s * val.x, s * val.y);
    }
  };
  fft_vector<L, S>(fft_smem + v * Shape<L>::LP, a.tw, a.tw_len / L, jt, in, out);
}

// type 2, correction + padding + y pass: KV columns i1 of f -> T[i1][y]
template <int L, int S>
__global__ void __launch_bounds__(Shape<L>::THREADS, Shape<L>::MIN_BLOCKS) fft_t2_cols_kernel(FusedArgs a) {
  extern __shared__ __align__(16) float2 fft_smem[];
  constexpr int KV = Shape<L>::KV;
  const int v = threadIdx.x % KV, jt = threadIdx.x / KV;
  const int i1 = blockIdx.x * KV + v;
  const bool ok = i1 < a.N1;
  const float2 *f = a.in + blockIdx.y * a.in_stride;
  float2 *trow = a.out + blockIdx.y * a.out_stride + (int64_t)(ok ? i1 : 0) * L;
  const float s1 = ok ? a.p1[i1] : 0.f;
  auto in = [&](int q) {
    const int i2 = mode_of(q, a.N2, a.h2, L);
    if (!ok || i2 < 0) return make_float2(0.f, 0.f);
    const float s = s1 * a.p2[i2];
    const float2 val = f[(int64_t)i2 * a.N1 + i1];
    return make_float2(s * val.x, s * val.y);
  };
  auto out = [&](int q, float2 val) {
    if (ok) trow[q] = val;
  };
  fft_vector<L, S>(fft_smem + v * Shape<L>::LP, a.tw, a.tw_len / L, jt, in, out);
}

// type 2, padding + x pass: KV columns y of T -> fine-grid rows y
template <int L, int S>
__global__ void __launch_bounds__(Shape<L>::THREADS, Shape<L>::MIN_BLOCKS) fft_t2_rows_kernel(FusedArgs a) {
  extern __shared__ __align__(16) float2 fft_smem[];
  constexpr int KV = Shape<L>::KV;
  const int v = threadIdx.x % KV, jt = threadIdx.x / KV;
  const int y = blockIdx.x * KV + v;
  const float2 *T = a.in + blockIdx.y * a.in_stride;
  float2 *row = a.out + blockIdx.y * a.out_stride + (int64_t)y * L;
  auto in = [&](int q) {
    const int i1 = mode_of(q, a.N1, a.h1, L);
    return i1 >= 0 ? T[(int64_t)i1 * a.n2 + y] : make_float2(0.f, 0.f);
  };
  auto out = [&](int q, float2 val) { row[q] = val; };
  fft_vector<L, S>(fft_smem + v * Shape<L>::LP, a.tw, a.tw_len / L, jt, in, out);
}

enum Pass { T1_ROWS, T1_COLS, T2_COLS, T2_ROWS };

template <int L, int S>
cudaError_t launch_pass(Pass pass, const FusedArgs &a, int nvec, cudaStream_t st) {
  void (*kern)(FusedArgs) = pass == T1_ROWS   ? fft_t1_rows_kernel<L, S>
                            : pass == T1_COLS ? fft_t1_cols_kernel<L, S>
                            : pass == T2_COLS ? fft_t2_cols_kernel<L, S>
                                              : fft_t2_rows_kernel<L, S>;
  const size_t smem = Shape<L>::SMEM;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // rows of the fine grid (x passes) or of T (y passes), KV per block
  const int vecs = (pass == T1_ROWS || pass == T2_ROWS) ? a.n2 : a.N1;
  const unsigned blocks = (unsigned)((vecs + Shape<L>::KV - 1) / Shape<L>::KV);
  kern<<<dim3(blocks, nvec), Shape<L>::THREADS, smem, st>>>(a);
  return cudaGetLastError();
}

template <int S>
cudaError_t launch_len(int L, Pass pass, const FusedArgs &a, int nvec, cudaStream_t st) {
  switch (L) {
    case 128: return launch_pass<128, S>(pass, a, nvec, st);
    case 256: return launch_pass<256, S>(pass, a, nvec, st);
    case 512: return launch_pass<512, S>(pass, a, nvec, st);
    case 1024: return launch_pass<1024, S>(pass, a, nvec, st);
    case 2048: return launch_pass<2048, S>(pass, a, nvec, st);
    case 4096: return launch_pass<4096, S>(pass, a, nvec, st);
    default: return cudaErrorInvalidValue;
  }
}

bool pow2_in_range(int64_t n) {
  return n >= (int64_t(1) << kMinLog) && n <= (int64_t(1) << kMaxLog) && (n & (n - 1)) == 0;
}

cudaError_t run_pass(const nufft_plan_s *p, Pass pass, const void *src, void *dst) {
  FusedArgs a{};
  a.in = static_cast<const float2 *>(src);
  a.out = static_cast<float2 *>(dst);
  a.grid = static_cast<float2 *>(p->grid);
  a.p1 = static_cast<const float *>(p->pfac[0]);
  a.p2 = static_cast<const float *>(p->pfac[1]);
  a.tw = static_cast<const float2 *>(p->fft_tw);
  a.tw_len = (int)std::max(p->n[0], p->n[1]);
  a.n1 = (int)p->n[0];
  a.n2 = (int)p->n[1];
  a.N1 = (int)p->N[0];
  a.N2 = (int)p->N[1];
  a.h1 = a.N1 / 2;
  a.h2 = a.N2 / 2;
  const int64_t grid = p->n[0] * p->n[1], work = p->N[0] * p->n[1], modes = p->N[0] * p->N[1];
  switch (pass) {
    case T1_ROWS: a.in_stride = grid; a.out_stride = work; break;
    case T1_COLS: a.in_stride = work; a.out_stride = modes; break;
    case T2_COLS: a.in_stride = modes; a.out_stride = work; break;
    case T2_ROWS: a.in_stride = work; a.out_stride = grid; break;
  }
  const int L = (pass == T1_ROWS || pass == T2_ROWS) ? a.n1 : a.n2;
  return p->iflag >= 0 ? launch_len<1>(L, pass, a, p->nvec, p->stream)
                       : launch_len<-1>(L, pass, a, p->nvec, p->stream);
}

}  // namespace

bool fused_fft_supported(const nufft_plan_s *p) {
  return p->dim == 2 && p->dtype == 0 && pow2_in_range(p->n[0]) && pow2_in_range(p->n[1]);
}

std::vector<float> fused_fft_twiddles(int64_t len, int sign) {
  // exp(s 2 pi i t / len) in double, rounded once to float
  std::vector<float> tw((size_t)(2 * len));
  const double two_pi = 6.283185307179586476925286766559;
  for (int64_t t = 0; t < len; t++) {
    const double ang = two_pi * (double)t / (double)len;
    tw[(size_t)(2 * t)] = (float)std::cos(ang);
    tw[(size_t)(2 * t + 1)] = (float)(sign * std::sin(ang));
  }
  return tw;
}

int64_t fused_fft_work_elems(const nufft_plan_s *p) { return p->N[0] * p->n[1]; }

cudaError_t launch_fused_t1(const nufft_plan_s *p, int stage, void *f) {
  return stage == 0 ? run_pass(p, T1_ROWS, p->grid, p->fft_work) : run_pass(p, T1_COLS, p->fft_work, f);
}

cudaError_t launch_fused_t2(const nufft_plan_s *p, int stage, const void *f) {
  return stage == 0 ? run_pass(p, T2_COLS, f, p->fft_work) : run_pass(p, T2_ROWS, p->fft_work, p->grid);
}

}  // namespace nufft
