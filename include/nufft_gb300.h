/*
 * nufft_gb300.h -- C ABI of the GB300 (sm_103a) nonuniform FFT library.
 *
 * Transforms (definitions from "cuFINUFFT: a load-balanced GPU library for
 * general-purpose nonuniform FFTs", Shih, Wright, Anden, Blaschke, Barnett;
 * section and equation numbers are that paper's):
 *
 *   type 1 (Sec. I eq. (1)):  f_k = sum_{j<M} c_j exp(s i k.x_j),   k in I_N1 x I_N2 (x I_N3)
 *   type 2 (Sec. I eq. (3)):  c_j = sum_k      f_k exp(s i k.x_j),  j < M
 *
 * with s = +1 if iflag >= 0, else -1, I_N = {k integer : -N/2 <= k < N/2}
 * (eq. (2)), and points x_j in [-pi, pi)^d (any finite value is accepted and
 * read modulo 2 pi).  They are computed approximately, to relative l2 error
 * close to eps, by the three-step scheme of Sec. II: spreading with the
 * "exponential of semicircle" kernel (eq. (5)) onto a fine grid of
 * n_i = 2 N_i points (eq. (7)), a plain FFT (eq. (9)), and truncation with
 * correction (eq. (10)); type 2 runs the transposed steps (eq. (11), (12),
 * Sec. II-B c).  No normalisation is applied.
 *
 * The interface follows the "plan, setup, execute, destroy" pattern of
 * Sec. I-A: one plan per (type, dim, modes, iflag, eps, precision); setpts
 * bin-sorts the points once (Sec. III-A) and any number of executes reuse
 * them with new strengths / coefficients.
 *
 * Conventions for every entry point
 *   - Return value: 0 (NUFFT_OK) on success, else a positive NUFFT_ERR_* code.
 *     No C++ exception crosses this interface.  nufft_strerror() names codes.
 *   - Complex arrays are interleaved (re, im) of the plan's real type:
 *     float for dtype 0 (complex64), double for dtype 1 (complex128).
 *   - Mode arrays f hold prod(N_i) values, k1 fastest, each k_i increasing
 *     from -floor(N_i/2).  Point arrays c hold M values in the caller's order.
 *   - Array pointers may be DEVICE memory (of the plan's device) or HOST
 *     memory (pinned or pageable).  Device pointers are used in place and the
 *     call is asynchronous on the plan's stream.  Host pointers are staged
 *     through plan-owned device buffers and the call returns only after the
 *     results have been copied back (synchronous).
 *   - The caller owns every array it passes; the library keeps no pointer to
 *     caller memory after a call returns.
 *   - Plans are not thread safe: one plan is used by one host thread at a time.
 */
#ifndef NUFFT_GB300_H
#define NUFFT_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct nufft_plan_s *nufft_plan_t;

/* Error codes (returned as int). */
#define NUFFT_OK 0
#define NUFFT_ERR_BAD_ARG 1        /* type, dim, N, iflag, dtype, NULL pointer, M < 0 */
#define NUFFT_ERR_BAD_EPS 2        /* eps <= 0, not finite, or width w outside [2, 16] */
#define NUFFT_ERR_ALLOC 3          /* device (or pinned host) allocation failed */
#define NUFFT_ERR_CUDA 4           /* a CUDA runtime call or kernel launch failed */
#define NUFFT_ERR_CUFFT 5          /* a cuFFT call failed */
#define NUFFT_ERR_NO_POINTS 6      /* execute before a successful setpts */
#define NUFFT_ERR_BAD_POINTS 7     /* a coordinate is NaN or infinite */
#define NUFFT_ERR_BAD_OPT 8        /* unknown option key or out-of-range value */
#define NUFFT_ERR_TOO_LARGE 9      /* sizes beyond the 32-bit index ranges used inside */

/* Indices of nufft_get_timings() output (milliseconds of the last execute /
 * setpts, measured with CUDA events on the plan's stream). */
#define NUFFT_T_SPREAD_INTERP 0    /* spreading (type 1) or interpolation (type 2) kernel */
#define NUFFT_T_FFT 1              /* fine-grid FFT: cuFFT execution; with the fused FFT, both of
                                      its passes (x and y), which include the correction */
#define NUFFT_T_DECONV_PAD 2       /* correction + truncation (type 1) or correction + padding (type 2);
                                      0 with the fused FFT, whose y pass does this work */
#define NUFFT_T_ZERO 3             /* clearing the fine grid before spreading (type 1) */
#define NUFFT_T_EXEC 4             /* whole execute on the device (first to last event) */
#define NUFFT_T_SETPTS 5           /* whole setpts on the device */
#define NUFFT_T_COUNT 6

/* Indices of nufft_get_info() output. */
#define NUFFT_I_W 0                /* kernel width w (eq. (6)) */
#define NUFFT_I_N1 1               /* fine grid n_1, n_2, n_3 (n_3 = 1 in 2D) */
#define NUFFT_I_N2 2
#define NUFFT_I_N3 3
#define NUFFT_I_M 4                /* points of the last setpts */
#define NUFFT_I_NBINS 5            /* number of bins */
#define NUFFT_I_NSUB 6             /* number of subproblems */
#define NUFFT_I_BIN1 7             /* bin size m_1, m_2, m_3 */
#define NUFFT_I_BIN2 8
#define NUFFT_I_BIN3 9
#define NUFFT_I_MSUB 10            /* points per subproblem cap M_sub */
#define NUFFT_I_METHOD 11          /* spreading method in use (NUFFT_METHOD_*) */
#define NUFFT_I_BATCH 12           /* vectors per pass of nufft_execute_batch */
#define NUFFT_I_FFT 13             /* 1: fused pruned FFT in use (option "fft"), 0: cuFFT */
#define NUFFT_I_SMS 14             /* multiprocessors of the plan's device (sizes the default M_sub) */
#define NUFFT_I_TILE3D 15          /* 3D REGTILE spreader in use: 1 planes per warp, 2 slab bins (0: not 3D) */
#define NUFFT_I_IGROUP 16          /* 3D single-precision SM interpolator: 1 one point per thread,
                                      K >= 2 points of one window origin per thread (0: other) */
#define NUFFT_I_BIN_ORIGIN 17      /* 1: points binned by window origin (the 3D slab spreader), 0: by cell */
#define NUFFT_I_COUNT 18

/* Spreading / interpolation methods (option "method"). */
#define NUFFT_METHOD_AUTO 0
#define NUFFT_METHOD_SM 1          /* Sec. III-A "SM": subproblems spread in shared memory */
#define NUFFT_METHOD_GM_SORT 2     /* Sec. III-A "GM-sort": thread per sorted point, global atomics */
#define NUFFT_METHOD_REGTILE 3     /* SM decomposition with the padded bin in registers (type 1) */
#define NUFFT_METHOD_GM 4          /* Sec. III-A/B "GM": thread per point in the caller's order, no sort */

/*
 * Create a plan.  Defined by Sec. I-A ("plan, setup, execute, destroy") and
 * Sec. II (parameters).
 *   type        1 or 2 (eq. (1) or eq. (3)).
 *   dim         1, 2 or 3 (1D: the definitions "in the obvious fashion", Sec. I).
 *   n_modes     host array of dim entries N_1, N_2 (, N_3), each >= 1.
 *   iflag       sign of the exponent: >= 0 -> +1, < 0 -> -1.
 *   eps         requested relative tolerance; sets the kernel width
 *               w = ceil(log10(1/eps)) + 1 and shape beta = 2.30 w (eq. (6)).
 *               Accepted when 2 <= w <= 16.
 *   dtype       0 = complex64 / float coordinates, 1 = complex128 / double.
 *   cuda_stream cudaStream_t to enqueue all work on (NULL: the legacy default
 *               stream).  The plan uses the device current at this call.
 *   out         receives the plan (set to NULL on failure).
 * Allocates the fine grid, the correction factors and the cuFFT plan on the
 * current device.  Errors: BAD_ARG, BAD_EPS, ALLOC, CUDA, CUFFT, TOO_LARGE.
 */
int nufft_makeplan(int type, int dim, const int64_t *n_modes, int iflag, double eps,
                   int dtype, void *cuda_stream, nufft_plan_t *out);

/*
 * nufft_makeplan with an upsampling factor sigma in (1, 2] instead of the
 * paper's fixed sigma = 2 (Sec. I-B, limitation 3, names smaller sigma as a way
 * to cut memory and run time; Sec. II gives the rule only for sigma = 2).
 * Rule used (eq. (6) at sigma = 2, and otherwise eq. (6) with the sigma
 * dependence of the ES kernel's error, which decays like
 * exp(-pi w sqrt(1 - 1/sigma))):
 *   w    = ceil(log10(1/eps) / sqrt(2 (1 - 1/sigma))) + 1,
 *   beta = 2.30 w (4/3) (1 - 1/(2 sigma)),
 *   n_i  = smallest 2^a 3^b 5^c >= max(sigma N_i, 2 w).
 * Products within 1e-9 of an integer count as that integer before a ceiling.
 * Smaller sigma means a smaller fine grid and FFT but a wider kernel.
 * Errors: as nufft_makeplan; BAD_ARG also for sigma outside (1, 2] or NaN;
 * BAD_EPS when the width comes out above 16.
 */
int nufft_makeplan_upsampled(int type, int dim, const int64_t *n_modes, int iflag, double eps,
                             int dtype, double sigma, void *cuda_stream, nufft_plan_t *out);

/*
 * Set a tuning option; takes effect at the next setpts.  Keys:
 *   "method"   NUFFT_METHOD_* (type 1 spreading; type 2 always uses the
 *              tiled shared-memory interpolator unless "method" is GM_SORT).
 *              AUTO picks REGTILE for type 1 and SM for type 2 (the only
 *              methods in 1D; others give BAD_OPT there).  REGTILE
 *              fixes the bin size (the "bin" options are ignored, except
 *              "bin2", the bin height, in 2D and 3D); it is a spreading
 *              method, so a type 2 plan given it runs as SM (info "method"
 *              then reads SM).
 *   "bin1", "bin2", "bin3"   bin size m_i in fine-grid cells (Sec. III-A), >= 1.
 *   "msub"     cap M_sub on points per subproblem (SM step 1), >= 1; at most
 *              8192 for 3D type 2 plans with the SM interpolator.
 *   "threads"  threads per block of the SM / GM-sort spreading and
 *              interpolation kernels (multiple of 32, 32..1024; lowered to
 *              what a kernel's register use allows).  Default 256; for the
 *              3D shared-memory interpolators 512 (complex64, one point per
 *              thread) and 1024 (complex128); the grouped complex64
 *              interpolator ("igroup") runs at most 256.
 *   "batch"    vectors per pass of nufft_execute_batch, 1..1024 (0: as many
 *              fine grids as fit in 1 GiB, at most 64).  Takes effect at the
 *              next execute.
 *   "regtile_cols"  tile columns per lane of the REGTILE spreader: 1, 2 or 4
 *              (0: 1).
 *   "tile3d"   3D REGTILE spreader: 1, one block per subproblem, each warp
 *              holding two padded planes of a bin of 32 - 2 ceil(w/2) x 8 x
 *              (16 - 2 ceil(w/2)) cells (16 x 4 x ... in double precision);
 *              2, one warp per subproblem holding the w planes of a bin one
 *              window origin thick in z (33 - w x 32 x 1 origins; complex64
 *              and w <= 8 only, else BAD_OPT at setpts).  With 2, setpts bins
 *              the points by window origin: the bin of a point is that of the
 *              node ceil(g - w/2) + floor(w/2) (its first support node shifted
 *              by floor(w/2)) instead of its cell floor(g) (info BIN_ORIGIN).
 *              0 (default): 2 where it applies, else 1.
 *   "igroup"   3D complex64 SM interpolation: 1, one thread per point; K = 2,
 *              3 or 4, the points of one window origin (the w^3 nodes they
 *              read) in groups of at most K per thread, each tile row loaded
 *              once per group.  setpts reorders the points of each
 *              subproblem by window origin and records the groups (w <= 8
 *              and the build's shared memory -- one counter per origin, 20
 *              bytes per point of M_sub -- within the device's limit, else
 *              BAD_OPT at setpts).  0 (default): 2 where it applies, else 1.
 *              Other plans ignore it.
 *   "fft"      0 (default): 2D complex64 plans whose fine grid sizes are
 *              powers of two from 128 to 4096 take the fine-grid FFT as two
 *              passes of the library's own kernels, pruned to the modes of
 *              I_N and fused with the correction of eq. (10) / (11); other
 *              plans use cuFFT.  1: always cuFFT and the separate correction
 *              kernels.
 * Errors: BAD_ARG (NULL), BAD_OPT (unknown key or invalid value).
 */
int nufft_set_opt(nufft_plan_t plan, const char *key, double value);

/*
 * Set the nonuniform points (Sec. III-A bin sort and SM step 1 subproblems).
 *   M        number of points, >= 0 (M = 0 makes execute produce zeros / nothing).
 *   x, y, z  M coordinates each, of the plan's real type; z is ignored (may be
 *            NULL) in 2D, y and z in 1D.  Host or device pointers.  Read once: the plan keeps
 *            its own sorted, grid-scaled copy, so the caller may free or
 *            overwrite them afterwards.
 * Synchronises the plan's stream once (to size the subproblem table).
 * Errors: BAD_ARG, BAD_POINTS (NaN/Inf coordinate), ALLOC, CUDA, TOO_LARGE.
 */
int nufft_setpts(nufft_plan_t plan, int64_t M, const void *x, const void *y, const void *z);

/*
 * Run the transform on the points of the last setpts.
 *   type 1: reads c (M complex), overwrites f (prod N_i complex).
 *   type 2: reads f, overwrites c.
 * Nothing is accumulated into the output.  Device pointers: asynchronous on
 * the plan's stream.  Host pointers: synchronous (see the conventions above).
 * Errors: BAD_ARG, NO_POINTS, ALLOC (host staging), CUDA, CUFFT.
 */
int nufft_execute(nufft_plan_t plan, void *c, void *f);

/*
 * Run the transform on nvec vectors with the points of the last setpts: the
 * reuse of sorted points "with new strength vectors" that motivates the
 * plan/setup/execute interface (cuFINUFFT paper, Sec. I).  Each vector is an
 * independent transform, exactly as nufft_execute would compute it.
 *   nvec   number of vectors, >= 0 (0: nothing happens).
 *   c      nvec * M complex, vector v at c + v M (type 1 input, type 2 output).
 *   f      nvec * prod N_i complex, vector v at f + v prod N_i.
 * Vectors go through the device in passes of "batch" vectors (info
 * NUFFT_I_BATCH): one zeroing / padding pass, one spreading / interpolation
 * launch, one batched cuFFT and one correction launch per pass (with the
 * fused FFT of option "fft": its two passes instead of the padding, cuFFT
 * and correction, and no zeroing when the previous pass left the grids
 * clear), over that many fine grids (allocated at the first execute that
 * needs them, kept by the plan).  Host and device pointers as for nufft_execute; host arrays go
 * through staging buffers of one pass.  Timings: stage times summed over the
 * passes, NUFFT_T_EXEC from the first pass's start to the last pass's end.
 * Errors: BAD_ARG, NO_POINTS, ALLOC (fine grids, staging), CUDA, CUFFT.
 */
int nufft_execute_batch(nufft_plan_t plan, int64_t nvec, void *c, void *f);

/* Release every resource of the plan (NULL is accepted).  Synchronises the
 * plan's stream first.  Errors: CUDA. */
int nufft_destroy(nufft_plan_t plan);

/*
 * Device times of the last execute and setpts, in milliseconds, indexed by
 * NUFFT_T_*.  Writes min(n, NUFFT_T_COUNT) doubles to the host array ms;
 * entries a plan's type does not have are 0.  Waits for the recorded events.
 * Errors: BAD_ARG, CUDA.
 */
int nufft_get_timings(nufft_plan_t plan, double *ms, int n);

/* Plan parameters, indexed by NUFFT_I_*; writes min(n, NUFFT_I_COUNT) values
 * to the host array info.  Errors: BAD_ARG. */
int nufft_get_info(nufft_plan_t plan, int64_t *info, int n);

/*
 * Copy the integer results of the last setpts to HOST arrays (for checking
 * the bin sort of Sec. III-A; any argument may be NULL to skip it):
 *   counts[nbins]     points per bin (bins ordered x fastest; a point's bin is
 *                     the bin of its cell, or of its window origin node
 *                     ceil(g - w/2) + floor(w/2) when info BIN_ORIGIN is 1);
 *   starts[nbins]     exclusive prefix sum of counts;
 *   perm[M]           the permutation t: sorted slot -> caller's point index
 *                     (points of bin 0, then bin 1, ...; order inside a bin is
 *                     unspecified);
 *   subprob[3*nsub]   (bin, first sorted slot, point count) per subproblem.
 * Synchronises the plan's stream.  Errors: BAD_ARG, NO_POINTS, BAD_OPT (the
 * GM method sorts nothing), CUDA.
 */
int nufft_get_sort(nufft_plan_t plan, int32_t *counts, int32_t *starts, int32_t *perm,
                   int32_t *subprob);

/*
 * Bin sort without any memory allocation.  The paper has no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc.  Examples are
 * hosts whose device memory is entirely reserved by their own pool allocator,
 * and real-time loops that must not pay allocation latency or risk
 * out-of-memory in the middle of a run.
 *
 * It computes what nufft_setpts computes for its counts and permutation: each
 * point's fine-grid cell and bin (bins of bins[i] cells, x fastest, smaller at
 * the far edge), the number of points per bin, and the permutation listing
 * the points of bin 0, then bin 1, ...  The order inside a bin is
 * unspecified.
 *   dim, dtype    2 or 3; 0 = float coordinates, 1 = double.
 *   M             number of points, 0 <= M <= 1,048,576.
 *   x, y, z       DEVICE arrays of M coordinates (z unused in 2D), read mod 2 pi.
 *   n_fine, bins  HOST arrays of dim fine-grid sizes and bin sizes (bins are
 *                 clamped to the grid).  At most 65,536 bins in total.
 *   counts        DEVICE output, one int32 per bin (overwritten).
 *   perm          DEVICE output, M int32 (overwritten).
 *   cuda_stream   stream to run on (NULL: legacy default stream).
 * Scratch: a fixed 8.3 MB array in the library's device memory, present on
 * every GPU that loads the library until the process exits.  The first call on
 * each device looks up that array's device address (once, with the device
 * current).  All calls share the one array: calls that overlap on the GPU
 * (different streams, or several host threads) race and must be serialised by
 * the caller.  The call blocks until the sort has finished: it ends by copying
 * an error flag to the host and synchronising the stream.
 * Calls no cudaMalloc, cudaFree or allocating library routine.
 * Errors: BAD_ARG, TOO_LARGE (M or the bin count above the limits),
 * BAD_POINTS (a NaN/Inf coordinate), CUDA.
 */
int nufft_binsort_noalloc(int dim, int dtype, int64_t M, const void *x, const void *y,
                          const void *z, const int64_t *n_fine, const int64_t *bins,
                          int32_t *counts, int32_t *perm, void *cuda_stream);

/* Static description of an error code. */
const char *nufft_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* NUFFT_GB300_H */
