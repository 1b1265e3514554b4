// Internal declarations of the GB300 NUFFT library: the plan object and the
// launchers each translation unit provides.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cufft.h>

#include <cstdint>
#include <utility>
#include <vector>

#include "../../include/nufft_gb300.h"

namespace nufft {

constexpr int kMaxDim = 3;
constexpr int kMinWidth = 2;
constexpr int kMaxWidth = 16;

// One subproblem of SM step 1 (Sec. III-A of the cuFINUFFT paper): a run of
// at most M_sub sorted points that all lie in one bin.
struct Subproblem {
  int32_t bin;
  int32_t start;  // first sorted slot
  int32_t count;  // number of points
  int32_t groups;  // grouped 3D single-precision interpolation: window-origin groups
                   // recorded for this subproblem (0 otherwise)
};

}  // namespace nufft

struct nufft_plan_s {
  // --- definition -------------------------------------------------------
  int type = 1;
  int dim = 2;
  int iflag = -1;
  int dtype = 0;  // 0 complex64, 1 complex128
  double eps = 0;
  double sigma = 2.0;  // upsampling factor
  int w = 0;
  double beta = 0;
  int64_t N[3] = {1, 1, 1};
  int64_t n[3] = {1, 1, 1};
  int device = 0;
  int num_sms = 1;             // multiprocessors of the device (queried at makeplan)
  cudaStream_t stream = nullptr;

  // --- options (applied at setpts) --------------------------------------
  int opt_method = NUFFT_METHOD_AUTO;
  int opt_bin[3] = {0, 0, 0};  // 0: default
  int opt_msub = 0;            // 0: default
  int opt_threads = 0;         // 0: default
  int opt_regtile_cols = 0;    // 0: default
  int opt_batch = 0;           // vectors per pass of a batched execute (0: default)
  int opt_fft = 0;             // 0: fused pruned FFT where supported, 1: cuFFT
  int opt_tile3d = 0;          // 3D register-tile spreader: 0 auto, 1 planes per warp, 2 slab bins
  int opt_igroup = 0;          // 3D single-precision SM interpolation: 0 auto, 1 one point per thread,
                               // 2..4 points sharing a window per thread

  // --- resolved at setpts ------------------------------------------------
  int method = NUFFT_METHOD_SM;
  int m[3] = {1, 1, 1};
  int nb[3] = {1, 1, 1};
  int msub = 1024;
  int threads = 256;
  int regtile_cols = 4;        // tile columns per lane of the register-tile spreader
  int tile3d = 1;              // 3D register-tile spreader in use: 1 planes per warp, 2 slab bins
  bool bin_origin = false;     // points binned by window origin (the slab spreader), not by cell
  int igroup = 0;              // 3D f32 SM interpolator in use: 1 one point per thread, K >= 2 groups
                               // of at most K points (0: another interpolator)
  int64_t nbins = 0;
  int64_t nsub = 0;
  int64_t M = 0;
  bool have_pts = false;
  int nvec = 1;                // vectors in the pass being launched (blockIdx.y range)
  bool fused_fft = false;      // fine-grid FFT by the fused pruned passes (fft2d_fused.cu)

  // --- device memory ----------------------------------------------------
  void *grid = nullptr;            // grid_vecs fine grids, each n1 n2 n3 complex, x fastest
  int64_t grid_vecs = 0;
  int64_t grid_zero_vecs = 0;      // leading fine grids known to be all zero (fused FFT clears them)
  void *pfac[3] = {nullptr, nullptr, nullptr};  // correction factors p_i(k), N_i reals
  int32_t *bin_counts = nullptr;   // nbins + 1
  int32_t *bin_starts = nullptr;   // nbins + 1 (last entry: M)
  int32_t *sub_counts = nullptr;   // nbins + 1
  int32_t *sub_starts = nullptr;   // nbins + 1
  int64_t cap_bins = 0;
  int32_t *cell_counts = nullptr;  // nbins * cells_per_bin + 1 (cell-level counting sort)
  int32_t *cell_starts = nullptr;  // same length: first sorted slot of each (bin, cell)
  int32_t *scan_scratch = nullptr; // block partials of the scans
  int64_t cap_keys = 0;
  int32_t *perm = nullptr;         // M: sorted slot -> user index
  void *gcoord[3] = {nullptr, nullptr, nullptr};  // M bin-relative grid coordinates
  int32_t *bin_of = nullptr;       // M (setpts scratch: each point's cell key)
  int32_t *rank_of = nullptr;      // M (setpts scratch)
  int64_t cap_pts = 0;
  void *gtmp = nullptr;            // setpts scratch: dim x M bin-relative coordinates, caller order
  int64_t cap_gtmp = 0;
  nufft::Subproblem *subprob = nullptr;
  uint32_t *grec = nullptr;        // grouped interpolation: one record per group, at the
  int64_t cap_grec = 0;            // sorted slots of its subproblem (interp_group3d_f32.cu)
  int64_t cap_sub = 0;
  int *flag = nullptr;             // device error flag (setpts)
  void *stage_c = nullptr;         // staging for host c
  int64_t cap_stage_c = 0;
  void *stage_f = nullptr;         // staging for host f
  int64_t cap_stage_f = 0;
  void *stage_xyz = nullptr;       // staging for host coordinates (3 M reals)
  int64_t cap_stage_xyz = 0;
  void *fft_tw = nullptr;          // fused FFT: exp(s 2 pi i t / max(n1, n2)), complex64
  void *fft_work = nullptr;        // fused FFT: N1 x n2 complex per vector of a pass
  int64_t cap_fft_work = 0;

  cufftHandle fft = 0;
  bool fft_made = false;
  std::vector<std::pair<int, cufftHandle>> fft_many;  // batched plans by vector count

  // --- timing -------------------------------------------------------------
  cudaEvent_t ev[8] = {};
  bool exec_recorded = false;
  std::vector<cudaEvent_t> xev;   // execute: 5 events per pass
  int xpasses = 0;                 // passes of the last execute
  bool setpts_recorded = false;
};

namespace nufft {

inline size_t real_size(const nufft_plan_s *p) { return p->dtype == 0 ? 4 : 8; }
inline int64_t grid_cells(const nufft_plan_s *p) { return p->n[0] * p->n[1] * p->n[2]; }
inline int64_t mode_count(const nufft_plan_s *p) { return p->N[0] * p->N[1] * p->N[2]; }

// setpts.cu: bin sort and subproblem table.  Returns a NUFFT_* code.
int run_setpts(nufft_plan_s *p, const void *x, const void *y, const void *z);
// setpts.cu: GM (unsorted) method: per-point cells and offsets only.
int run_setpts_gm(nufft_plan_s *p, const void *x, const void *y, const void *z);

// spreadinterp_*.cu: type 1 spreading (grid must be zeroed) and type 2
// interpolation, for the plan's dim, dtype and width.
// Explicitly instantiated in spreadinterp_{2,3}d_{f32,f64}.cu.
template <int DIM, typename T>
cudaError_t launch_spread_t(const nufft_plan_s *p, const void *c);
template <int DIM, typename T>
cudaError_t launch_interp_t(const nufft_plan_s *p, void *c);

// Register-tile 2D spreader (spread_regtile.cuh), instantiated in
// spread_regtile_{f32,f64}.cu, and the bin size it is built for.
template <typename T>
cudaError_t launch_spread_regtile2d(const nufft_plan_s *p, const void *c);
void regtile2d_bins(int w, int cols, int *m1, int *m2);
// Register-tile 3D spreader (spread_plane3d.cuh), instantiated in
// spread_plane3d_{f32,f64}.cu, and the bin size it is built for.
template <typename T>
cudaError_t launch_spread_plane3d(const nufft_plan_s *p, const void *c);
void plane3d_bins(int w, int dtype, int *m1, int *m2, int *m3);
// 3D single-precision spreader with one-cell-thick bins (spread_slab3d.cuh),
// for widths up to kSlab3DMaxWidth ((w+1)^2 complex accumulators per lane).
constexpr int kSlab3DMaxWidth = 8;
bool slab3d_supported(int w, int dtype);
void slab3d_bins(int w, int *m1, int *m2, int *m3);
cudaError_t launch_spread_slab3d(const nufft_plan_s *p, const void *c);
// 3D single-precision interpolation with tile reads shared by points of one
// window origin (interp_group3d_f32.cu): supported for w <= kGroup3DMaxWidth
// when its shared memory fits (p->m and p->msub resolved), group size p->igroup.
constexpr int kGroup3DMaxWidth = 8;
constexpr int kGroup3DDefault = 2;  // option sweep: 2.42 ms (K = 2), 2.46 (3, 4), 3.20 (1)
bool group3d_supported(const nufft_plan_s *p, int smem_max);
cudaError_t build_groups3d(const nufft_plan_s *p);
cudaError_t launch_interp_group3d(const nufft_plan_s *p, void *c);

// spreadinterp_1d.cu: 1D register-tile spreading and shared-memory interpolation.
cudaError_t launch_spread_1d(const nufft_plan_s *p, const void *c);
cudaError_t launch_interp_1d(const nufft_plan_s *p, void *c);

// deconv.cu: type 1 correction + truncation, type 2 correction + padding.
cudaError_t launch_deconvolve(const nufft_plan_s *p, void *f);
cudaError_t launch_pad(const nufft_plan_s *p, const void *f);

// fft2d_fused.cu: the fine-grid FFT of 2D complex64 plans whose fine grid
// sizes are powers of two in 256..4096, pruned to the kept modes and fused
// with the correction steps.  Type 1: stage 0 is the x pass (grid ->
// workspace; it leaves the pass's fine grids zeroed), stage 1 the y pass with
// the correction (workspace -> f).
// Type 2: stage 0 is the correction, padding and y pass (f -> workspace),
// stage 1 the x pass (workspace -> grid).
bool fused_fft_supported(const nufft_plan_s *p);
std::vector<float> fused_fft_twiddles(int64_t len, int sign);  // interleaved re, im
int64_t fused_fft_work_elems(const nufft_plan_s *p);           // complex per vector
cudaError_t launch_fused_t1(const nufft_plan_s *p, int stage, void *f);
cudaError_t launch_fused_t2(const nufft_plan_s *p, int stage, const void *f);

// scan.cu: exclusive prefix sum of n int32 values; out has n + 1 entries and
// out[n] receives the total.  scratch holds scan_scratch_len(n) ints.
int64_t scan_scratch_len(int64_t n);
cudaError_t exclusive_scan(const int32_t *in, int32_t *out, int64_t n, int32_t *scratch,
                           cudaStream_t s);

}  // namespace nufft
