// Plan object and C ABI of the GB300 NUFFT library (declared in
// include/nufft_gb300.h).
//
// Source: "cuFINUFFT: a load-balanced GPU library for general-purpose
// nonuniform FFTs" (Shih, Wright, Anden, Blaschke, Barnett).  The plan holds
// the parameters of Sec. II (width and shape from eq. (6), fine grid sizes,
// correction factors of eq. (10)), the fine grid, the cuFFT plan used for
// eq. (9) / (12), and the bin-sort results of Sec. III-A that setpts
// produces; execute runs the three steps on the plan's stream.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "nufft_internal.cuh"

using nufft::real_size;

namespace {

constexpr double kPi = 3.14159265358979323846;

// ---------------------------------------------------------------- parameters

// A value within 1e-9 (relative) of an integer is taken as that integer, so
// decimal tolerances and factors do not flip a ceiling on rounding noise
// (1e-6 gives log10 = 6 exactly, hence w = 7).
double snap_int(double v) {
  const double r = std::nearbyint(v);
  return std::fabs(v - r) <= 1e-9 * std::max(1.0, std::fabs(v)) ? r : v;
}

// Kernel width: eq. (6), w = ceil(log10(1/eps)) + 1, at sigma = 2.  For
// sigma < 2 the digit count is stretched by 1 / sqrt(2 (1 - 1/sigma)), the
// ratio of the ES kernel's error exponents pi w sqrt(1 - 1/sigma) at sigma = 2
// and at sigma (the paper fixes sigma = 2 and gives no rule for other values).
int width_for(double eps, double sigma) {
  const double L = snap_int(-std::log10(eps));
  if (sigma == 2.0) return (int)std::ceil(L) + 1;
  return (int)std::ceil(snap_int(L / std::sqrt(2.0 * (1.0 - 1.0 / sigma)))) + 1;
}

// Kernel shape: eq. (6), beta = 2.30 w, at sigma = 2; for sigma < 2 scaled by
// (1 - 1/(2 sigma)) / (3/4), the ES kernel's optimal-shape dependence.
double beta_for(int w, double sigma) {
  if (sigma == 2.0) return 2.30 * w;
  return 2.30 * w * (4.0 / 3.0) * (1.0 - 0.5 / sigma);
}

// Smallest 2^a 3^b 5^c >= v.
int64_t next_smooth(int64_t v) {
  for (int64_t n = v < 1 ? 1 : v;; n++) {
    int64_t m = n;
    for (int64_t f : {2, 3, 5})
      while (m % f == 0) m /= f;
    if (m == 1) return n;
  }
}

// Gauss-Legendre rule on [-1, 1] by Newton iteration on P_q.
void gauss_legendre(int q, std::vector<double> &x, std::vector<double> &wts) {
  x.resize(q);
  wts.resize(q);
  for (int i = 0; i < q; i++) {
    double t = std::cos(kPi * (4.0 * i + 3.0) / (4.0 * q + 2.0));
    double p_q = 0, p_q1 = 0;
    for (int it = 0; it < 100; it++) {
      double a = 1.0, b = t;  // P_0, P_1
      for (int k = 2; k <= q; k++) {
        const double c = ((2 * k - 1) * t * b - (k - 1) * a) / k;
        a = b;
        b = c;
      }
      p_q = b;
      p_q1 = a;
      const double dp = q * (t * p_q - p_q1) / (t * t - 1.0);
      const double step = p_q / dp;
      t -= step;
      if (std::fabs(step) < 1e-16) break;
    }
    double a = 1.0, b = t;
    for (int k = 2; k <= q; k++) {
      const double c = ((2 * k - 1) * t * b - (k - 1) * a) / k;
      a = b;
      b = c;
    }
    const double dp = q * (t * b - a) / (t * t - 1.0);
    x[i] = t;
    wts[i] = 2.0 / ((1.0 - t * t) * dp * dp);
  }
}

// Correction factors p(k) = (2/w) / phihat(alpha k), alpha = w pi / n, for the
// modes k of I_N in increasing order (text after eq. (10)).  phihat is the
// Fourier transform (eq. (4)) of the ES kernel (eq. (5)),
//   phihat(xi) = 2 int_0^1 exp(beta (sqrt(1 - z^2) - 1)) cos(xi z) dz,
// taken with z = sin(theta) so that the integrand is smooth:
//   2 int_0^{pi/2} exp(beta (cos theta - 1)) cos(xi sin theta) cos theta dtheta.
std::vector<double> correction_factors(int64_t N, int64_t n, int w, double beta) {
  std::vector<double> gx, gw;
  gauss_legendre(100, gx, gw);
  std::vector<double> th(gx.size()), wt(gx.size());
  for (size_t i = 0; i < gx.size(); i++) {
    th[i] = (gx[i] + 1.0) * (kPi / 4.0);
    wt[i] = gw[i] * (kPi / 4.0) * std::exp(beta * (std::cos(th[i]) - 1.0)) * std::cos(th[i]);
  }
  const double alpha = w * kPi / (double)n;
  std::vector<double> p((size_t)N);
  const int64_t kmin = -(N / 2);
  for (int64_t i = 0; i < N; i++) {
    const double xi = alpha * (double)(kmin + i);
    double s = 0.0;
    for (size_t q = 0; q < th.size(); q++) s += wt[q] * std::cos(xi * std::sin(th[q]));
    p[(size_t)i] = (2.0 / w) / (2.0 * s);
  }
  return p;
}

// ---------------------------------------------------------------- helpers

bool is_device_ptr(const void *ptr, int device, bool *ok) {
  cudaPointerAttributes attr;
  *ok = true;
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error state
    return false;       // unknown to CUDA: pageable host memory
  }
  if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged) {
    if (attr.type == cudaMemoryTypeDevice && attr.device != device) *ok = false;
    return true;
  }
  return false;  // pinned or unregistered host memory
}

int grow_buffer(void **buf, int64_t *cap, int64_t bytes) {
  if (*buf && *cap >= bytes) return NUFFT_OK;
  if (*buf) cudaFree(*buf);
  *buf = nullptr;
  *cap = 0;
  if (cudaMalloc(buf, (size_t)(bytes > 0 ? bytes : 16)) != cudaSuccess) {
    cudaGetLastError();
    return NUFFT_ERR_ALLOC;
  }
  *cap = bytes;
  return NUFFT_OK;
}

// Default bin sizes.  2D: the padded bin of the interpolator is 32 x 32
// cells (bins 32 - 2 ceil(w/2) square; Sec. III-A Remark 1 found 32 x 32 bins
// best on its GPU).  3D: the largest bins, halving the longest side, whose
// padded tile fits the shared-memory budget.
void default_bins(const nufft_plan_s *p, int m[3]) {
  const int pad = (p->w + 1) / 2;
  const size_t cs = 2 * real_size(p);
  if (p->dim == 2) {
    m[0] = m[1] = 32 - 2 * pad;
    m[2] = 1;
  } else {
    m[0] = m[1] = 16;
    m[2] = 8;
    const size_t budget = p->dtype == 0 ? 96 * 1024 : 200 * 1024;
    for (;;) {
      const size_t bytes = (size_t)(m[0] + 2 * pad) * (m[1] + 2 * pad) * (m[2] + 2 * pad) * cs;
      if (bytes <= budget || (m[0] == 1 && m[1] == 1 && m[2] == 1)) break;
      int d = 0;
      for (int i = 1; i < 3; i++)
        if (m[i] > m[d]) d = i;
      m[d] = (m[d] + 1) / 2;
    }
  }
}

size_t tile_bytes(const nufft_plan_s *p, const int m[3]) {
  const int pad = (p->w + 1) / 2;
  size_t cells = 1;
  for (int d = 0; d < p->dim; d++) cells *= (size_t)(m[d] + 2 * pad);
  return cells * 2 * real_size(p);
}

void release(nufft_plan_s *p) {
  cudaFree(p->grid);
  for (int d = 0; d < 3; d++) {
    cudaFree(p->pfac[d]);
    cudaFree(p->gcoord[d]);
  }
  cudaFree(p->bin_counts);
  cudaFree(p->bin_starts);
  cudaFree(p->sub_counts);
  cudaFree(p->sub_starts);
  cudaFree(p->scan_scratch);
  cudaFree(p->cell_counts);
  cudaFree(p->cell_starts);
  cudaFree(p->perm);
  cudaFree(p->bin_of);
  cudaFree(p->rank_of);
  cudaFree(p->gtmp);
  cudaFree(p->subprob);
  cudaFree(p->grec);
  cudaFree(p->flag);
  cudaFree(p->stage_c);
  cudaFree(p->stage_f);
  cudaFree(p->stage_xyz);
  cudaFree(p->fft_tw);
  cudaFree(p->fft_work);
  if (p->fft_made) cufftDestroy(p->fft);
  for (auto &h : p->fft_many) cufftDestroy(h.second);
  for (auto &e : p->xev) cudaEventDestroy(e);
  for (auto &e : p->ev)  // also the ones made before a failed makeplan
    if (e) cudaEventDestroy(e);
}

int cuda_code(cudaError_t e) {
  if (e == cudaSuccess) return NUFFT_OK;
  if (e == cudaErrorMemoryAllocation) return NUFFT_ERR_ALLOC;
  return NUFFT_ERR_CUDA;
}

// Event slots: setpts in ev[]; execute uses kPassEvents per pass in xev
// (type 1: zero, spread, FFT, deconvolve, end; type 2: pad, FFT, interp, end).
enum { EV_SET0 = 6, EV_SET1 = 7 };
constexpr int kPassEvents = 5;

// Vectors per pass of a batched execute: the "batch" option, else as many
// fine grids as fit in 1 GiB (at least 1, at most 64).
int64_t batch_pass(const nufft_plan_s *p) {
  if (p->opt_batch > 0) return p->opt_batch;
  const int64_t grid_bytes = nufft::grid_cells(p) * 2 * (int64_t)nufft::real_size(p);
  return std::max<int64_t>(1, std::min<int64_t>(64, (int64_t(1) << 30) / grid_bytes));
}

// cuFFT plan transforming nv consecutive fine grids.
int fft_plan_for(nufft_plan_s *p, int nv, cufftHandle *out) {
  if (nv == 1) {
    *out = p->fft;
    return NUFFT_OK;
  }
  for (auto &h : p->fft_many)
    if (h.first == nv) {
      *out = h.second;
      return NUFFT_OK;
    }
  int dims[3];
  for (int d = 0; d < p->dim; d++) dims[d] = (int)p->n[p->dim - 1 - d];  // slowest first
  const int dist = (int)nufft::grid_cells(p);
  cufftHandle h;
  const cufftResult r = cufftPlanMany(&h, p->dim, dims, nullptr, 1, dist, nullptr, 1, dist,
                                      p->dtype == 0 ? CUFFT_C2C : CUFFT_Z2Z, nv);
  if (r != CUFFT_SUCCESS) return r == CUFFT_ALLOC_FAILED ? NUFFT_ERR_ALLOC : NUFFT_ERR_CUFFT;
  if (cufftSetStream(h, p->stream) != CUFFT_SUCCESS) {
    cufftDestroy(h);
    return NUFFT_ERR_CUFFT;
  }
  p->fft_many.emplace_back(nv, h);
  *out = h;
  return NUFFT_OK;
}

}  // namespace

// ==================================================================== C ABI

extern "C" {

const char *nufft_strerror(int code) {
  switch (code) {
    case NUFFT_OK: return "success";
    case NUFFT_ERR_BAD_ARG: return "invalid argument";
    case NUFFT_ERR_BAD_EPS: return "tolerance out of range (kernel width must be 2..16)";
    case NUFFT_ERR_ALLOC: return "memory allocation failed";
    case NUFFT_ERR_CUDA: return "CUDA runtime error";
    case NUFFT_ERR_CUFFT: return "cuFFT error";
    case NUFFT_ERR_NO_POINTS: return "execute called before a successful setpts";
    case NUFFT_ERR_BAD_POINTS: return "a point coordinate is NaN or infinite";
    case NUFFT_ERR_BAD_OPT: return "unknown option or invalid option value";
    case NUFFT_ERR_TOO_LARGE: return "problem size beyond the supported index range";
    default: return "unknown error code";
  }
}

int nufft_makeplan(int type, int dim, const int64_t *n_modes, int iflag, double eps, int dtype,
                   void *cuda_stream, nufft_plan_t *out) {
  return nufft_makeplan_upsampled(type, dim, n_modes, iflag, eps, dtype, 2.0, cuda_stream, out);
}

int nufft_makeplan_upsampled(int type, int dim, const int64_t *n_modes, int iflag, double eps,
                             int dtype, double sigma, void *cuda_stream, nufft_plan_t *out) {
  if (out) *out = nullptr;
  if (!out || !n_modes || (type != 1 && type != 2) || dim < 1 || dim > 3 ||
      (dtype != 0 && dtype != 1) || !(sigma > 1.0 && sigma <= 2.0))
    return NUFFT_ERR_BAD_ARG;
  for (int d = 0; d < dim; d++)
    if (n_modes[d] < 1) return NUFFT_ERR_BAD_ARG;
  if (!(eps > 0) || !std::isfinite(eps)) return NUFFT_ERR_BAD_EPS;
  const int w = width_for(eps, sigma);
  if (w < nufft::kMinWidth || w > nufft::kMaxWidth) return NUFFT_ERR_BAD_EPS;

  nufft_plan_s *p = new (std::nothrow) nufft_plan_s();
  if (!p) return NUFFT_ERR_ALLOC;
  p->type = type;
  p->dim = dim;
  p->iflag = iflag >= 0 ? 1 : -1;
  p->dtype = dtype;
  p->eps = eps;
  p->w = w;
  p->beta = beta_for(w, sigma);
  p->sigma = sigma;
  int64_t cells = 1, modes = 1;
  for (int d = 0; d < dim; d++) {
    p->N[d] = n_modes[d];
    if (p->N[d] > (int64_t(1) << 29)) {
      delete p;
      return NUFFT_ERR_TOO_LARGE;
    }
    // fine grid: smallest 2^a 3^b 5^c >= max(sigma N_i, 2 w) (Sec. II, after eq. (6))
    const int64_t sn = (int64_t)std::ceil(snap_int(sigma * (double)p->N[d]));
    p->n[d] = next_smooth(std::max<int64_t>(sn, 2 * (int64_t)w));
    cells *= p->n[d];
    modes *= p->N[d];
  }
  if (cells > (int64_t(1) << 36) || modes > (int64_t(1) << 34)) {
    delete p;
    return NUFFT_ERR_TOO_LARGE;
  }
  p->stream = static_cast<cudaStream_t>(cuda_stream);
  int rc = NUFFT_OK;
  do {
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
      rc = NUFFT_ERR_CUDA;
      break;
    }
    const size_t rs = real_size(p);
    if (cudaMalloc(&p->grid, (size_t)cells * 2 * rs) != cudaSuccess) { rc = NUFFT_ERR_ALLOC; break; }
    p->grid_vecs = 1;
    for (int d = 0; d < 3; d++) {
      // dimensions beyond dim get the single factor 1, so the 2D correction
      // kernels serve 1D plans unchanged
      std::vector<double> pf = d < dim ? correction_factors(p->N[d], p->n[d], w, p->beta)
                                       : std::vector<double>(1, 1.0);
      if (cudaMalloc(&p->pfac[d], pf.size() * rs) != cudaSuccess) { rc = NUFFT_ERR_ALLOC; break; }
      cudaError_t e;
      if (dtype == 0) {
        std::vector<float> pf32(pf.begin(), pf.end());
        e = cudaMemcpy(p->pfac[d], pf32.data(), pf32.size() * 4, cudaMemcpyHostToDevice);
      } else {
        e = cudaMemcpy(p->pfac[d], pf.data(), pf.size() * 8, cudaMemcpyHostToDevice);
      }
      if (e != cudaSuccess) { rc = NUFFT_ERR_CUDA; break; }
    }
    if (rc) break;
    if (nufft::fused_fft_supported(p)) {
      const std::vector<float> tw = nufft::fused_fft_twiddles(std::max(p->n[0], p->n[1]), p->iflag);
      if (cudaMalloc(&p->fft_tw, tw.size() * 4) != cudaSuccess) { rc = NUFFT_ERR_ALLOC; break; }
      if (cudaMemcpy(p->fft_tw, tw.data(), tw.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
        rc = NUFFT_ERR_CUDA;
        break;
      }
    }
    // cuFFT: row-major dims, slowest first (our x index is fastest)
    cufftResult fr;
    const cufftType ft = dtype == 0 ? CUFFT_C2C : CUFFT_Z2Z;
    if (dim == 1)
      fr = cufftPlan1d(&p->fft, (int)p->n[0], ft, 1);
    else if (dim == 2)
      fr = cufftPlan2d(&p->fft, (int)p->n[1], (int)p->n[0], ft);
    else
      fr = cufftPlan3d(&p->fft, (int)p->n[2], (int)p->n[1], (int)p->n[0], ft);
    if (fr != CUFFT_SUCCESS) { rc = fr == CUFFT_ALLOC_FAILED ? NUFFT_ERR_ALLOC : NUFFT_ERR_CUFFT; break; }
    p->fft_made = true;
    if (cufftSetStream(p->fft, p->stream) != CUFFT_SUCCESS) { rc = NUFFT_ERR_CUFFT; break; }
    for (auto &e : p->ev)
      if (cudaEventCreate(&e) != cudaSuccess) { rc = NUFFT_ERR_CUDA; break; }
    if (rc) break;
  } while (false);
  if (rc) {
    cudaGetLastError();
    release(p);
    delete p;
    return rc;
  }
  *out = p;
  return NUFFT_OK;
}

int nufft_set_opt(nufft_plan_t p, const char *key, double value) {
  if (!p || !key) return NUFFT_ERR_BAD_ARG;
  if (!std::isfinite(value) || value != std::floor(value)) return NUFFT_ERR_BAD_OPT;
  const int64_t v = (int64_t)value;
  if (!std::strcmp(key, "method")) {
    if (v != NUFFT_METHOD_AUTO && v != NUFFT_METHOD_SM && v != NUFFT_METHOD_GM_SORT &&
        v != NUFFT_METHOD_REGTILE && v != NUFFT_METHOD_GM)
      return NUFFT_ERR_BAD_OPT;
    p->opt_method = (int)v;
  } else if (!std::strcmp(key, "bin1") || !std::strcmp(key, "bin2") || !std::strcmp(key, "bin3")) {
    if (v < 0 || v > 4096) return NUFFT_ERR_BAD_OPT;
    p->opt_bin[key[3] - '1'] = (int)v;
  } else if (!std::strcmp(key, "msub")) {
    if (v < 0 || v > (int64_t(1) << 24)) return NUFFT_ERR_BAD_OPT;
    p->opt_msub = (int)v;
  } else if (!std::strcmp(key, "batch")) {
    if (v != 0 && (v < 1 || v > 1024 || v != (double)(int)v)) return NUFFT_ERR_BAD_OPT;
    p->opt_batch = (int)v;
  } else if (!std::strcmp(key, "fft")) {
    if (v != 0 && v != 1) return NUFFT_ERR_BAD_OPT;
    p->opt_fft = (int)v;
  } else if (!std::strcmp(key, "regtile_cols")) {
    if (v != 0 && v != 1 && v != 2 && v != 4) return NUFFT_ERR_BAD_OPT;
    p->opt_regtile_cols = (int)v;
  } else if (!std::strcmp(key, "tile3d")) {
    if (v < 0 || v > 2) return NUFFT_ERR_BAD_OPT;
    p->opt_tile3d = (int)v;
  } else if (!std::strcmp(key, "igroup")) {
    if (v < 0 || v > 4) return NUFFT_ERR_BAD_OPT;
    p->opt_igroup = (int)v;
  } else if (!std::strcmp(key, "threads")) {
    if (v != 0 && (v < 32 || v > 1024 || v % 32)) return NUFFT_ERR_BAD_OPT;
    p->opt_threads = (int)v;
  } else {
    return NUFFT_ERR_BAD_OPT;
  }
  return NUFFT_OK;
}

int nufft_setpts(nufft_plan_t p, int64_t M, const void *x, const void *y, const void *z) {
  if (!p || M < 0 || (M > 0 && (!x || (p->dim >= 2 && !y) || (p->dim == 3 && !z))))
    return NUFFT_ERR_BAD_ARG;
  if (M > (int64_t(1) << 31) - 1) return NUFFT_ERR_TOO_LARGE;
  p->have_pts = false;
  if (cudaSetDevice(p->device) != cudaSuccess) return NUFFT_ERR_CUDA;

  // resolve options
  p->method = p->opt_method;
  if (p->method == NUFFT_METHOD_AUTO)
    p->method = p->type == 1 ? NUFFT_METHOD_REGTILE : NUFFT_METHOD_SM;
  // the register tile is a spreading scheme: a type 2 plan runs as SM
  if (p->type == 2 && p->method == NUFFT_METHOD_REGTILE) p->method = NUFFT_METHOD_SM;
  // 1D: register-tile spreading and shared-memory interpolation only
  if (p->dim == 1 && p->method != NUFFT_METHOD_REGTILE && p->method != NUFFT_METHOD_SM)
    return NUFFT_ERR_BAD_OPT;
  if (p->dim == 1) p->method = p->type == 1 ? NUFFT_METHOD_REGTILE : NUFFT_METHOD_SM;
  int m[3];
  default_bins(p, m);
  for (int d = 0; d < 3; d++)
    if (d < p->dim && p->opt_bin[d] > 0) m[d] = p->opt_bin[d];
  p->regtile_cols = p->opt_regtile_cols > 0 ? p->opt_regtile_cols : 1;
  p->bin_origin = false;
  if (p->dim == 1) {
    // one padded-bin column per lane for spreading; long bins for the
    // interpolator's staged tile, short enough in single precision that the
    // bin-relative coordinate keeps ~1e-6 cell resolution (double: 512 cells,
    // from the option sweep of the 1D double-precision workload)
    m[0] = p->type == 1 ? 32 - 2 * ((p->w + 1) / 2) : (p->dtype == 0 ? 128 : 512);
    if (p->opt_bin[0] > 0 && p->type == 2) m[0] = p->opt_bin[0];
  } else if (p->method == NUFFT_METHOD_REGTILE) {
    if (p->dim == 2) {
      nufft::regtile2d_bins(p->w, p->regtile_cols, &m[0], &m[1]);
      if (p->opt_bin[1] > 0) m[1] = p->opt_bin[1];  // rows are free
    } else {
      // planes per warp (1) or one-cell-thick slab bins (2, single precision,
      // w <= 8; the default where it applies: 4.84 against 5.84 ms on the 3D
      // single-precision workload)
      const bool slab_ok = nufft::slab3d_supported(p->w, p->dtype);
      if (p->opt_tile3d == 2 && !slab_ok) return NUFFT_ERR_BAD_OPT;
      p->tile3d = p->opt_tile3d == 1 ? 1 : (slab_ok ? 2 : 1);
      p->bin_origin = p->tile3d == 2;  // the slab spreader bins points by window origin
      if (p->tile3d == 2)
        nufft::slab3d_bins(p->w, &m[0], &m[1], &m[2]);
      else
        nufft::plane3d_bins(p->w, p->dtype, &m[0], &m[1], &m[2]);
      if (p->opt_bin[1] > 0) m[1] = p->opt_bin[1];  // rows are free
    }
  }
  for (int d = 0; d < 3; d++) {
    if (d >= p->dim) m[d] = 1;
    if (m[d] > p->n[d]) m[d] = (int)p->n[d];
  }
  int smem_max = 0;
  if (cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  if (p->method == NUFFT_METHOD_SM && tile_bytes(p, m) > (size_t)smem_max) return NUFFT_ERR_BAD_OPT;
  p->nbins = 1;
  for (int d = 0; d < 3; d++) {
    p->m[d] = m[d];
    p->nb[d] = (int)((p->n[d] + m[d] - 1) / m[d]);
    p->nbins *= p->nb[d];
  }
  if (p->opt_msub > 0) {
    p->msub = p->opt_msub;
  } else if (p->method == NUFFT_METHOD_REGTILE) {
    // a subproblem is one warp (2D) or one block (3D) walking rows in order:
    // cap it so that small problems still spread over every SM (32 warps or
    // 4 blocks per SM).  Caps from the option sweeps: 512 points in 2D, 8192
    // in 3D single precision, 2048 for the two-float 3D spreader
    // (slab bins: 4096, one subproblem per bin at the bench density -- a bin
    // split in several subproblems flushes its rows once per subproblem)
    const bool warp_sub = p->dim <= 2 || p->tile3d == 2;  // one warp per subproblem
    const int64_t cap = p->dim <= 2 ? 512 : (p->tile3d == 2 ? 4096 : (p->dtype == 0 ? 8192 : 2048));
    const int64_t fill = M / ((int64_t)p->num_sms * (warp_sub ? 32 : 4));
    p->msub = (int)std::max<int64_t>(64, std::min<int64_t>(cap, fill));
  } else {
    // interpolation: 4096 points in 3D (single precision: one subproblem per
    // 16 x 16 x 8 bin at the bench density, fuller buckets for its
    // bank-spread point order) and for the long 1D double-precision bins,
    // 2048 otherwise (option sweeps)
    p->msub = p->type == 2 ? (p->dim == 3 || (p->dim == 1 && p->dtype == 1) ? 4096 : 2048) : 1024;
  }
  // the 3D shared-memory interpolator keeps a per-block order of its points
  // next to the tile (single precision; the cap applies to both)
  if (p->dim == 3 && p->type == 2 && p->method == NUFFT_METHOD_SM && p->msub > 8192) p->msub = 8192;
  // GM packs a point's cell index into int32
  if (p->method == NUFFT_METHOD_GM && nufft::grid_cells(p) >= (int64_t(1) << 31)) return NUFFT_ERR_TOO_LARGE;
  // the cell-level sort indexes (bin, cell) pairs with int32
  if (p->nbins * (int64_t)m[0] * m[1] * m[2] >= (int64_t(1) << 31) - 1) return NUFFT_ERR_TOO_LARGE;
  // 3D single-precision SM interpolation: points grouped by window origin
  // where the kernel's shared memory fits (the default), else one point per
  // thread
  p->igroup = 0;
  if (p->dim == 3 && p->type == 2 && p->method == NUFFT_METHOD_SM && p->dtype == 0) {
    const bool ok = nufft::group3d_supported(p, smem_max);
    if (p->opt_igroup >= 2 && !ok) return NUFFT_ERR_BAD_OPT;
    p->igroup = p->opt_igroup == 1 ? 1 : (p->opt_igroup >= 2 ? p->opt_igroup : (ok ? nufft::kGroup3DDefault : 1));
  }
  // the 3D interpolators hold one large tile per block (two blocks per SM in
  // single precision, one in double): more threads per block keep more warps
  // per SM busy (512 and 1024 from the option sweeps); the grouped kernel
  // holds K points' weights per thread and runs 256
  const int def_threads = (p->dim == 3 && p->type == 2 && p->method == NUFFT_METHOD_SM)
                              ? (p->dtype == 0 ? (p->igroup >= 2 ? 256 : 512) : 1024)
                              : 256;
  p->threads = p->opt_threads > 0 ? p->opt_threads : def_threads;
  p->fused_fft = p->opt_fft == 0 && p->fft_tw != nullptr;
  p->M = M;

  // coordinates in host memory are staged through a device buffer
  const void *xyz[3] = {x, p->dim >= 2 ? y : nullptr, p->dim == 3 ? z : nullptr};
  if (M > 0) {
    const size_t bytes = (size_t)M * real_size(p);
    for (int d = 0; d < p->dim; d++) {
      bool ok;
      if (is_device_ptr(xyz[d], p->device, &ok)) {
        if (!ok) return NUFFT_ERR_BAD_ARG;
        continue;
      }
      int rc = grow_buffer(&p->stage_xyz, &p->cap_stage_xyz, (int64_t)(3 * bytes));
      if (rc) return rc;
      void *dst = static_cast<char *>(p->stage_xyz) + d * bytes;
      if (cudaMemcpyAsync(dst, xyz[d], bytes, cudaMemcpyHostToDevice, p->stream) != cudaSuccess)
        return NUFFT_ERR_CUDA;
      xyz[d] = dst;
    }
  }
  if (cudaEventRecord(p->ev[EV_SET0], p->stream) != cudaSuccess) return NUFFT_ERR_CUDA;
  const int rc = p->method == NUFFT_METHOD_GM ? nufft::run_setpts_gm(p, xyz[0], xyz[1], xyz[2])
                                              : nufft::run_setpts(p, xyz[0], xyz[1], xyz[2]);
  if (rc) {
    cudaGetLastError();
    return rc;
  }
  if (cudaEventRecord(p->ev[EV_SET1], p->stream) != cudaSuccess) return NUFFT_ERR_CUDA;
  p->setpts_recorded = true;
  p->have_pts = true;
  return NUFFT_OK;
}

int nufft_execute(nufft_plan_t p, void *c, void *f) { return nufft_execute_batch(p, 1, c, f); }

int nufft_execute_batch(nufft_plan_t p, int64_t nvec, void *c, void *f) {
  if (!p || nvec < 0) return NUFFT_ERR_BAD_ARG;
  if (!p->have_pts) return NUFFT_ERR_NO_POINTS;
  if (nvec == 0) return NUFFT_OK;
  if (!f || (p->M > 0 && !c)) return NUFFT_ERR_BAD_ARG;
  if (cudaSetDevice(p->device) != cudaSuccess) return NUFFT_ERR_CUDA;
  cudaStream_t s = p->stream;
  const size_t cb = 2 * real_size(p);
  const int64_t cells = nufft::grid_cells(p), modes = nufft::mode_count(p);
  const size_t c_bytes = (size_t)p->M * cb, f_bytes = (size_t)modes * cb;
  const int64_t pass = std::min<int64_t>(nvec, batch_pass(p));
  const int64_t npass = (nvec + pass - 1) / pass;

  bool ok = true;
  const bool c_host = p->M > 0 && !is_device_ptr(c, p->device, &ok);
  if (!ok) return NUFFT_ERR_BAD_ARG;
  const bool f_host = !is_device_ptr(f, p->device, &ok);
  if (!ok) return NUFFT_ERR_BAD_ARG;
  int rc = NUFFT_OK;
  if (c_host && (rc = grow_buffer(&p->stage_c, &p->cap_stage_c, (int64_t)(pass * c_bytes)))) return rc;
  if (f_host && (rc = grow_buffer(&p->stage_f, &p->cap_stage_f, (int64_t)(pass * f_bytes)))) return rc;
  // fine grids for one pass (the old ones are freed only once the new fit)
  if (p->grid_vecs < pass) {
    void *g = nullptr;
    if (cudaMalloc(&g, (size_t)(pass * cells) * cb) != cudaSuccess) {
      cudaGetLastError();
      return NUFFT_ERR_ALLOC;
    }
    cudaFree(p->grid);
    p->grid = g;
    p->grid_vecs = pass;
    p->grid_zero_vecs = 0;
  }
  if (p->fused_fft &&
      (rc = grow_buffer(&p->fft_work, &p->cap_fft_work, (int64_t)(pass * nufft::fused_fft_work_elems(p) * cb))))
    return rc;
  while ((int64_t)p->xev.size() < npass * kPassEvents) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return NUFFT_ERR_CUDA;
    p->xev.push_back(e);
  }

  const int dir = p->iflag >= 0 ? CUFFT_INVERSE : CUFFT_FORWARD;
  p->exec_recorded = false;
  cudaError_t e = cudaSuccess;
  for (int64_t k = 0; k < npass; k++) {
    const int64_t v0 = k * pass, nv = std::min<int64_t>(pass, nvec - v0);
    char *cu = static_cast<char *>(c) + (c ? v0 * c_bytes : 0);  // caller's arrays of this pass
    char *fu = static_cast<char *>(f) + v0 * f_bytes;
    void *dc = c_host ? p->stage_c : cu, *df = f_host ? p->stage_f : fu;
    if (p->type == 1 && c_host && cudaMemcpyAsync(dc, cu, nv * c_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return NUFFT_ERR_CUDA;
    if (p->type == 2 && f_host && cudaMemcpyAsync(df, fu, nv * f_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return NUFFT_ERR_CUDA;
    cufftHandle plan_fft = 0;
    if (!p->fused_fft && (rc = fft_plan_for(p, (int)nv, &plan_fft))) return rc;
    p->nvec = (int)nv;
    cudaEvent_t *ev = &p->xev[k * kPassEvents];
    auto fft = [&]() -> int {
      cufftResult r = p->dtype == 0
                          ? cufftExecC2C(plan_fft, (cufftComplex *)p->grid, (cufftComplex *)p->grid, dir)
                          : cufftExecZ2Z(plan_fft, (cufftDoubleComplex *)p->grid,
                                         (cufftDoubleComplex *)p->grid, dir);
      return r == CUFFT_SUCCESS ? NUFFT_OK : NUFFT_ERR_CUFFT;
    };
    auto spread = [&]() -> cudaError_t {
      if (p->M == 0 || (p->method != NUFFT_METHOD_GM && p->nsub == 0)) return cudaSuccess;
      if (p->dim == 1) return nufft::launch_spread_1d(p, dc);
      if (p->method == NUFFT_METHOD_REGTILE && p->dim == 2)
        return p->dtype == 0 ? nufft::launch_spread_regtile2d<float>(p, dc)
                             : nufft::launch_spread_regtile2d<double>(p, dc);
      if (p->method == NUFFT_METHOD_REGTILE && p->tile3d == 2) return nufft::launch_spread_slab3d(p, dc);
      if (p->method == NUFFT_METHOD_REGTILE)
        return p->dtype == 0 ? nufft::launch_spread_plane3d<float>(p, dc)
                             : nufft::launch_spread_plane3d<double>(p, dc);
      if (p->dim == 2)
        return p->dtype == 0 ? nufft::launch_spread_t<2, float>(p, dc) : nufft::launch_spread_t<2, double>(p, dc);
      return p->dtype == 0 ? nufft::launch_spread_t<3, float>(p, dc) : nufft::launch_spread_t<3, double>(p, dc);
    };
    auto interp = [&]() -> cudaError_t {
      if (p->M == 0 || (p->method != NUFFT_METHOD_GM && p->nsub == 0)) return cudaSuccess;
      if (p->dim == 1) return nufft::launch_interp_1d(p, dc);
      if (p->igroup >= 2) return nufft::launch_interp_group3d(p, dc);
      if (p->dim == 2)
        return p->dtype == 0 ? nufft::launch_interp_t<2, float>(p, dc) : nufft::launch_interp_t<2, double>(p, dc);
      return p->dtype == 0 ? nufft::launch_interp_t<3, float>(p, dc) : nufft::launch_interp_t<3, double>(p, dc);
    };
    if (p->type == 1) {
      // zero -> spread (eq. (7)) -> FFT (eq. (9)) -> correct + truncate (eq. (10));
      // fused: x pass, then y pass with the correction.  The fused x pass
      // leaves the grids it read zeroed, so the clear is skipped after it.
      const bool zeroed = p->fused_fft && p->grid_zero_vecs >= nv;
      p->grid_zero_vecs = 0;
      if ((e = cudaEventRecord(ev[0], s)) != cudaSuccess ||
          (!zeroed && (e = cudaMemsetAsync(p->grid, 0, (size_t)(nv * cells) * cb, s)) != cudaSuccess) ||
          (e = cudaEventRecord(ev[1], s)) != cudaSuccess || (e = spread()) != cudaSuccess ||
          (e = cudaEventRecord(ev[2], s)) != cudaSuccess)
        break;
      if (p->fused_fft ? (e = nufft::launch_fused_t1(p, 0, df)) != cudaSuccess : (rc = fft()) != NUFFT_OK) break;
      if (p->fused_fft) p->grid_zero_vecs = nv;
      if ((e = cudaEventRecord(ev[3], s)) != cudaSuccess ||
          (e = p->fused_fft ? nufft::launch_fused_t1(p, 1, df) : nufft::launch_deconvolve(p, df)) != cudaSuccess ||
          (e = cudaEventRecord(ev[4], s)) != cudaSuccess)
        break;
    } else {
      // correct + pad (eq. (11)) -> FFT (eq. (12)) -> interpolate (Sec. II-B c);
      // fused: correction, padding and y pass, then x pass
      if ((e = cudaEventRecord(ev[0], s)) != cudaSuccess) break;
      if (p->M > 0 && (e = p->fused_fft ? nufft::launch_fused_t2(p, 0, df) : nufft::launch_pad(p, df)) != cudaSuccess)
        break;
      if ((e = cudaEventRecord(ev[1], s)) != cudaSuccess) break;
      if (p->M > 0 && (p->fused_fft ? (e = nufft::launch_fused_t2(p, 1, df)) != cudaSuccess : (rc = fft()) != NUFFT_OK))
        break;
      if ((e = cudaEventRecord(ev[2], s)) != cudaSuccess || (e = interp()) != cudaSuccess ||
          (e = cudaEventRecord(ev[3], s)) != cudaSuccess)
        break;
    }
    // host results of this pass
    if (p->type == 1 && f_host && cudaMemcpyAsync(fu, df, nv * f_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return NUFFT_ERR_CUDA;
    if (p->type == 2 && c_host && cudaMemcpyAsync(cu, dc, nv * c_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return NUFFT_ERR_CUDA;
    p->xpasses = (int)(k + 1);
  }
  p->nvec = 1;
  if (rc) return rc;
  if (e != cudaSuccess) return cuda_code(e);
  p->exec_recorded = true;
  if ((c_host || f_host) && cudaStreamSynchronize(s) != cudaSuccess) return NUFFT_ERR_CUDA;
  return NUFFT_OK;
}

int nufft_destroy(nufft_plan_t p) {
  if (!p) return NUFFT_OK;
  cudaSetDevice(p->device);
  const cudaError_t e = cudaStreamSynchronize(p->stream);
  release(p);
  delete p;
  return e == cudaSuccess ? NUFFT_OK : NUFFT_ERR_CUDA;
}

int nufft_get_timings(nufft_plan_t p, double *ms, int n) {
  if (!p || !ms || n < 0) return NUFFT_ERR_BAD_ARG;
  double t[NUFFT_T_COUNT] = {0, 0, 0, 0, 0, 0};
  auto span = [&](cudaEvent_t a, cudaEvent_t b, double *dst) -> int {
    float v = 0;
    if (cudaEventSynchronize(b) != cudaSuccess) return NUFFT_ERR_CUDA;
    if (cudaEventElapsedTime(&v, a, b) != cudaSuccess) return NUFFT_ERR_CUDA;
    *dst += v;
    return NUFFT_OK;
  };
  int rc;
  if (p->exec_recorded) {
    // stage times summed over the passes of the last execute; the fused FFT's
    // y pass (which holds the correction) counts as FFT time
    const int last = p->type == 1 ? 4 : 3;
    const int cor = p->fused_fft ? NUFFT_T_FFT : NUFFT_T_DECONV_PAD;
    const int stage[2][4] = {{NUFFT_T_ZERO, NUFFT_T_SPREAD_INTERP, NUFFT_T_FFT, cor},
                             {cor, NUFFT_T_FFT, NUFFT_T_SPREAD_INTERP, -1}};
    for (int k = 0; k < p->xpasses; k++) {
      cudaEvent_t *ev = &p->xev[k * kPassEvents];
      for (int i = 0; i < last; i++)
        if ((rc = span(ev[i], ev[i + 1], &t[stage[p->type - 1][i]]))) return rc;
    }
    if ((rc = span(p->xev[0], p->xev[(p->xpasses - 1) * kPassEvents + last], &t[NUFFT_T_EXEC]))) return rc;
  }
  if (p->setpts_recorded && (rc = span(p->ev[EV_SET0], p->ev[EV_SET1], &t[NUFFT_T_SETPTS]))) return rc;
  for (int i = 0; i < n && i < NUFFT_T_COUNT; i++) ms[i] = t[i];
  return NUFFT_OK;
}

int nufft_get_info(nufft_plan_t p, int64_t *info, int n) {
  if (!p || !info || n < 0) return NUFFT_ERR_BAD_ARG;
  const int64_t v[NUFFT_I_COUNT] = {p->w,    p->n[0], p->n[1], p->n[2], p->M,      p->nbins,  p->nsub,
                                    p->m[0], p->m[1], p->m[2], p->msub, p->method, batch_pass(p),
                                    p->fused_fft ? 1 : 0, p->num_sms, p->dim == 3 ? p->tile3d : 0, p->igroup,
                                    p->bin_origin ? 1 : 0};
  for (int i = 0; i < n && i < NUFFT_I_COUNT; i++) info[i] = v[i];
  return NUFFT_OK;
}

int nufft_get_sort(nufft_plan_t p, int32_t *counts, int32_t *starts, int32_t *perm, int32_t *subprob) {
  if (!p) return NUFFT_ERR_BAD_ARG;
  if (!p->have_pts) return NUFFT_ERR_NO_POINTS;
  if (p->method == NUFFT_METHOD_GM) return NUFFT_ERR_BAD_OPT;
  if (cudaSetDevice(p->device) != cudaSuccess || cudaStreamSynchronize(p->stream) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  const size_t nb = (size_t)p->nbins * 4;
  if (counts && cudaMemcpy(counts, p->bin_counts, nb, cudaMemcpyDeviceToHost) != cudaSuccess) return NUFFT_ERR_CUDA;
  if (starts && cudaMemcpy(starts, p->bin_starts, nb, cudaMemcpyDeviceToHost) != cudaSuccess) return NUFFT_ERR_CUDA;
  if (perm && p->M > 0 && cudaMemcpy(perm, p->perm, (size_t)p->M * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return NUFFT_ERR_CUDA;
  if (subprob && p->nsub > 0) {
    std::vector<nufft::Subproblem> tmp((size_t)p->nsub);
    if (cudaMemcpy(tmp.data(), p->subprob, tmp.size() * sizeof(nufft::Subproblem), cudaMemcpyDeviceToHost) !=
        cudaSuccess)
      return NUFFT_ERR_CUDA;
    for (size_t i = 0; i < tmp.size(); i++) {
      subprob[3 * i] = tmp[i].bin;
      subprob[3 * i + 1] = tmp[i].start;
      subprob[3 * i + 2] = tmp[i].count;
    }
  }
  return NUFFT_OK;
}

}  // extern "C"
