/*
 * Oracle for the 2D/3D type 1 and type 2 nonuniform FFT: plain, slow, double
 * precision C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * path.
 *
 * Source: "cuFINUFFT: a load-balanced GPU library for general-purpose
 * nonuniform FFTs" (Shih, Wright, Anden, Blaschke, Barnett), cited below as
 * [cuFINUFFT].  Section and equation numbers are that paper's.
 *
 * Contents
 *   - direct sums of eq. (1) (type 1) and eq. (3) (type 2), for all modes or a
 *     chosen subset (definition, not an approximation);
 *   - step 1 of type 1 (spreading, eq. (7)-(8)) and step 3 of type 2
 *     (interpolation, Sec. II-B c), one point after another, in user order;
 *   - the point-to-bin assignment and stable counting sort of Sec. III-A
 *     (GM-sort / SM precomputation), and the subproblem split of SM step 1;
 *   - Gauss-Legendre nodes for the kernel Fourier transform quadrature.
 * The FFT (eq. (9), (12)) and the diagonal correction (eq. (10), (11)) are
 * done in oracle/__init__.py with numpy, between these loops.
 *
 * Compiled with -ffp-contract=off so that no multiply-add is fused: the
 * fine-grid coordinate, which decides integer bin and cell indices, must be
 * rounded operation by operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* the double nearest to pi */
#define ORACLE_PI 3.14159265358979323846

/* ---------------------------------------------------------------------- */
/* Direct sums (O1)                                                        */
/* ---------------------------------------------------------------------- */

/* Compensated (Kahan) accumulation of one complex sum. */
typedef struct { double sr, cr, si, ci; } ksum;

static void ksum_add(ksum *s, double vr, double vi) {
    double y = vr - s->cr;
    double t = s->sr + y;
    s->cr = (t - s->sr) - y;
    s->sr = t;
    y = vi - s->ci;
    t = s->si + y;
    s->ci = (t - s->si) - y;
    s->si = t;
}

/*
 * Type 1 by definition, [cuFINUFFT] Sec. I eq. (1) (and its 1D and 3D
 * analogues, "in the obvious fashion"; y and z are unused in 1D, z in 2D):
 *   f_k = sum_j c_j exp(s i (k1 x_j + k2 y_j + k3 z_j)),  s = +1 if iflag >= 0
 *   else -1 (eq. (1) itself is s = -1),
 * on the tensor grid of modes K1 x K2 (x K3): the nk_i integers listed in
 * k1s, k2s (k3s).  exp(s i k.x) is the product of the per-dimension factors
 * exp(s i k_d x_d), each from its own cos and sin.  f: interleaved complex,
 * k1 fastest, nk1 * nk2 (* nk3) entries; c: M interleaved complex.
 */
void oracle_direct_type1(int dim, int64_t M, const double *x, const double *y,
                         const double *z, const double *c, int iflag,
                         int64_t nk1, const int64_t *k1s, int64_t nk2,
                         const int64_t *k2s, int64_t nk3, const int64_t *k3s,
                         double *f) {
    double s = iflag >= 0 ? 1.0 : -1.0;
    if (dim <= 2) nk3 = 1;
    if (dim == 1) nk2 = 1;
    int64_t nk = nk1 * nk2 * nk3;
    ksum *acc = (ksum *)calloc((size_t)nk, sizeof(ksum));
    double *e1 = (double *)malloc(sizeof(double) * 2 * (size_t)nk1);
    double *e2 = (double *)malloc(sizeof(double) * 2 * (size_t)nk2);
    double *e3 = (double *)malloc(sizeof(double) * 2 * (size_t)nk3);
    for (int64_t j = 0; j < M; j++) {
        for (int64_t a = 0; a < nk1; a++) {
            double ph = (double)k1s[a] * x[j];
            e1[2 * a] = cos(ph);
            e1[2 * a + 1] = s * sin(ph);
        }
        for (int64_t a = 0; a < nk2; a++) {
            double ph = dim >= 2 ? (double)k2s[a] * y[j] : 0.0;
            e2[2 * a] = cos(ph);
            e2[2 * a + 1] = s * sin(ph);
        }
        for (int64_t a = 0; a < nk3; a++) {
            double ph = dim == 3 ? (double)k3s[a] * z[j] : 0.0;
            e3[2 * a] = cos(ph);
            e3[2 * a + 1] = s * sin(ph);
        }
        double cr = c[2 * j], ci = c[2 * j + 1];
        for (int64_t i3 = 0; i3 < nk3; i3++) {
            /* c_j * e3 */
            double ar = cr * e3[2 * i3] - ci * e3[2 * i3 + 1];
            double ai = cr * e3[2 * i3 + 1] + ci * e3[2 * i3];
            for (int64_t i2 = 0; i2 < nk2; i2++) {
                double br = ar * e2[2 * i2] - ai * e2[2 * i2 + 1];
                double bi = ar * e2[2 * i2 + 1] + ai * e2[2 * i2];
                ksum *row = acc + nk1 * (i2 + nk2 * i3);
                for (int64_t i1 = 0; i1 < nk1; i1++) {
                    double er = e1[2 * i1], ei = e1[2 * i1 + 1];
                    ksum_add(&row[i1], br * er - bi * ei, br * ei + bi * er);
                }
            }
        }
    }
    for (int64_t q = 0; q < nk; q++) {
        f[2 * q] = acc[q].sr;
        f[2 * q + 1] = acc[q].si;
    }
    free(acc);
    free(e1);
    free(e2);
    free(e3);
}

/*
 * Type 2 by definition, [cuFINUFFT] Sec. I eq. (3):
 *   c_j = sum_{k in I_N1 x I_N2 (x I_N3)} f_k exp(s i (k . x_j)),
 * s = +1 if iflag >= 0 else -1 (eq. (3) itself is s = +1).
 * f is in mode order k1 fastest, each k_i running over I_N (eq. (2)), i.e.
 * from -floor(N_i/2) upwards.  Only the targets listed in `targets` (nt user
 * indices) are evaluated; c_out[q] belongs to targets[q].  The sum over k is
 * taken dimension by dimension (k1 innermost), each factor exp(s i k_d x_d)
 * from its own cos and sin.
 */
void oracle_direct_type2(int dim, const int64_t *N, const double *x,
                         const double *y, const double *z, const double *f,
                         int iflag, int64_t nt, const int64_t *targets,
                         double *c_out) {
    double s = iflag >= 0 ? 1.0 : -1.0;
    int64_t N1 = N[0], N2 = dim >= 2 ? N[1] : 1, N3 = dim == 3 ? N[2] : 1;
    int64_t k1min = -(N1 / 2), k2min = -(N2 / 2), k3min = -(N3 / 2);
    double *e1 = (double *)malloc(sizeof(double) * 2 * (size_t)N1);
    double *e2 = (double *)malloc(sizeof(double) * 2 * (size_t)N2);
    double *e3 = (double *)malloc(sizeof(double) * 2 * (size_t)N3);
    for (int64_t q = 0; q < nt; q++) {
        int64_t j = targets[q];
        for (int64_t i = 0; i < N1; i++) {
            double ph = (double)(k1min + i) * x[j];
            e1[2 * i] = cos(ph);
            e1[2 * i + 1] = s * sin(ph);
        }
        for (int64_t i = 0; i < N2; i++) {
            double ph = dim >= 2 ? (double)(k2min + i) * y[j] : 0.0;
            e2[2 * i] = cos(ph);
            e2[2 * i + 1] = s * sin(ph);
        }
        for (int64_t i = 0; i < N3; i++) {
            double ph = dim == 3 ? (double)(k3min + i) * z[j] : 0.0;
            e3[2 * i] = cos(ph);
            e3[2 * i + 1] = s * sin(ph);
        }
        ksum s3 = {0, 0, 0, 0};
        for (int64_t i3 = 0; i3 < N3; i3++) {
            ksum s2 = {0, 0, 0, 0};
            for (int64_t i2 = 0; i2 < N2; i2++) {
                ksum s1 = {0, 0, 0, 0};
                const double *row = f + 2 * N1 * (i2 + N2 * i3);
                for (int64_t i1 = 0; i1 < N1; i1++) {
                    double fr = row[2 * i1], fi = row[2 * i1 + 1];
                    double er = e1[2 * i1], ei = e1[2 * i1 + 1];
                    ksum_add(&s1, fr * er - fi * ei, fr * ei + fi * er);
                }
                double er = e2[2 * i2], ei = e2[2 * i2 + 1];
                ksum_add(&s2, s1.sr * er - s1.si * ei, s1.sr * ei + s1.si * er);
            }
            double er = e3[2 * i3], ei = e3[2 * i3 + 1];
            ksum_add(&s3, s2.sr * er - s2.si * ei, s2.sr * ei + s2.si * er);
        }
        c_out[2 * q] = s3.sr;
        c_out[2 * q + 1] = s3.si;
    }
    free(e1);
    free(e2);
    free(e3);
}

/* ---------------------------------------------------------------------- */
/* Fine grid geometry                                                      */
/* ---------------------------------------------------------------------- */

/*
 * Fine-grid coordinate of a point, [cuFINUFFT] eq. (7): node l of the fine
 * grid sits at l*h, h = 2 pi / n.  The sum is 2 pi periodic in x, so x is
 * first reduced to one period [0, 2 pi) (counted in turns), then scaled by n.
 * Returns g in [0, n); floor(g) is the cell the point lies in.
 */
double oracle_grid_coord(double x, int64_t n) {
    const double inv_two_pi = 1.0 / (2.0 * ORACLE_PI);
    double t = x * inv_two_pi;
    t = t - floor(t);
    double g = t * (double)n;
    if (g >= (double)n) g -= (double)n;
    return g;
}

/* ES kernel, [cuFINUFFT] eq. (5): exp(beta (sqrt(1 - z^2) - 1)) on |z| <= 1. */
static double es_kernel(double z, double beta) {
    if (fabs(z) > 1.0) return 0.0;
    return exp(beta * (sqrt(1.0 - z * z) - 1.0));
}

/*
 * The w fine-grid nodes a point at fine coordinate g touches, and their kernel
 * weights.  With psi(x) = phi(x / alpha), alpha = w pi / n (eq. (8)), the
 * weight of node l is phi((l h - x) / alpha) = phi((l - g) * 2 / w).  The
 * nodes taken are l0 .. l0 + w - 1 with l0 = ceil(g - w/2): every node with
 * z in [-1, 1).
 */
static int64_t support(double g, int w, double beta, double *ker) {
    int64_t l0 = (int64_t)ceil(g - 0.5 * (double)w);
    for (int t = 0; t < w; t++) {
        double zz = ((double)(l0 + t) - g) * 2.0 / (double)w;
        ker[t] = es_kernel(zz, beta);
    }
    return l0;
}

static int64_t wrap(int64_t l, int64_t n) {
    int64_t r = l % n;
    return r < 0 ? r + n : r;
}

/* ---------------------------------------------------------------------- */
/* Spreading and interpolation (steps of O2)                               */
/* ---------------------------------------------------------------------- */

/*
 * Type 1 step 1 (spreading), [cuFINUFFT] Sec. II-A eq. (7):
 *   b_l = sum_j c_j psi_per(l1 h1 - x_j, l2 h2 - y_j [, l3 h3 - z_j]),
 * accumulated one point at a time in user order.  b is the fine grid, n1 x n2
 * (x n3), x index fastest, interleaved complex, and is overwritten.
 */
void oracle_spread(int dim, const int64_t *n, int w, double beta, int64_t M,
                   const double *x, const double *y, const double *z,
                   const double *c, double *b) {
    int64_t n1 = n[0], n2 = dim >= 2 ? n[1] : 1, n3 = dim == 3 ? n[2] : 1;
    memset(b, 0, sizeof(double) * 2 * (size_t)(n1 * n2 * n3));
    double k1[32], k2[32], k3[32];
    int w2 = dim >= 2 ? w : 1;
    for (int64_t j = 0; j < M; j++) {
        int64_t a1 = support(oracle_grid_coord(x[j], n1), w, beta, k1);
        int64_t a2 = 0;
        k2[0] = 1.0;
        if (dim >= 2) a2 = support(oracle_grid_coord(y[j], n2), w, beta, k2);
        int64_t a3 = 0;
        int w3 = 1;
        k3[0] = 1.0;
        if (dim == 3) {
            a3 = support(oracle_grid_coord(z[j], n3), w, beta, k3);
            w3 = w;
        }
        double cr = c[2 * j], ci = c[2 * j + 1];
        for (int t3 = 0; t3 < w3; t3++) {
            int64_t l3 = dim == 3 ? wrap(a3 + t3, n3) : 0;
            for (int t2 = 0; t2 < w2; t2++) {
                int64_t l2 = dim >= 2 ? wrap(a2 + t2, n2) : 0;
                for (int t1 = 0; t1 < w; t1++) {
                    int64_t l1 = wrap(a1 + t1, n1);
                    double wt = k1[t1] * k2[t2] * k3[t3];
                    int64_t idx = l1 + n1 * (l2 + n2 * l3);
                    b[2 * idx] += wt * cr;
                    b[2 * idx + 1] += wt * ci;
                }
            }
        }
    }
}

/*
 * Type 2 step 3 (interpolation), [cuFINUFFT] Sec. II-B c:
 *   c_j = sum_l b_l psi_per(l1 h1 - x_j, l2 h2 - y_j [, l3 h3 - z_j]),
 * the transpose of oracle_spread.  c is overwritten (M interleaved complex).
 */
void oracle_interp(int dim, const int64_t *n, int w, double beta, int64_t M,
                   const double *x, const double *y, const double *z,
                   const double *b, double *c) {
    int64_t n1 = n[0], n2 = dim >= 2 ? n[1] : 1, n3 = dim == 3 ? n[2] : 1;
    double k1[32], k2[32], k3[32];
    int w2 = dim >= 2 ? w : 1;
    for (int64_t j = 0; j < M; j++) {
        int64_t a1 = support(oracle_grid_coord(x[j], n1), w, beta, k1);
        int64_t a2 = 0;
        k2[0] = 1.0;
        if (dim >= 2) a2 = support(oracle_grid_coord(y[j], n2), w, beta, k2);
        int64_t a3 = 0;
        int w3 = 1;
        k3[0] = 1.0;
        if (dim == 3) {
            a3 = support(oracle_grid_coord(z[j], n3), w, beta, k3);
            w3 = w;
        }
        double sr = 0.0, si = 0.0;
        for (int t3 = 0; t3 < w3; t3++) {
            int64_t l3 = dim == 3 ? wrap(a3 + t3, n3) : 0;
            for (int t2 = 0; t2 < w2; t2++) {
                int64_t l2 = dim >= 2 ? wrap(a2 + t2, n2) : 0;
                for (int t1 = 0; t1 < w; t1++) {
                    int64_t l1 = wrap(a1 + t1, n1);
                    double wt = k1[t1] * k2[t2] * k3[t3];
                    int64_t idx = l1 + n1 * (l2 + n2 * l3);
                    sr += wt * b[2 * idx];
                    si += wt * b[2 * idx + 1];
                }
            }
        }
        c[2 * j] = sr;
        c[2 * j + 1] = si;
    }
}

/* ---------------------------------------------------------------------- */
/* Bin sort and subproblems (integer setpts results)                       */
/* ---------------------------------------------------------------------- */

/*
 * [cuFINUFFT] Sec. III-A (GM-sort): the fine grid is cut into bins of
 * m1 x m2 (x m3) cells (smaller at the far edge), ordered x fastest.  A point
 * is in the bin holding its cell floor(g_i) in every dimension.  bin_of[j] is
 * that bin; counts[b] the number of points in bin b; starts[b] the exclusive
 * prefix sum of counts; perm the permutation t listing the points of bin 0,
 * then bin 1, ..., each bin's points in increasing user index (a stable
 * counting sort; the paper leaves the order inside a bin open).
 * Returns the number of bins.
 */
/*
 * The grid index a point is binned by: its cell floor(g) (w == 0, the
 * paper's bin of a point), or, with w > 0, the node l0 + floor(w/2) (mod n)
 * where l0 = ceil(g - w/2) is the first node of its support (support()
 * above): the bin then holds the point's window origin shifted by
 * floor(w/2), so the window lies inside the bin padded by floor(w/2) nodes
 * on the left and w - 1 - floor(w/2) on the right.  l0 + floor(w/2) =
 * ceil(g - oc) with oc = w/2 - floor(w/2) (1/2 or 0); it is evaluated in
 * that form, where no rounding enters (g - 3, say, rounds for g below about
 * 2e-16 and would move such a point's node by one).
 */
static int64_t bin_index(double x, int64_t n, int w) {
    const double g = oracle_grid_coord(x, n);
    if (w == 0) return (int64_t)floor(g);
    const double oc = 0.5 * (double)w - (double)(w / 2);
    return wrap((int64_t)ceil(g - oc), n);
}

static int64_t binsort_by(int dim, const int64_t *n, const int64_t *m, int w, int64_t M,
                          const double *x, const double *y, const double *z,
                          int32_t *bin_of, int32_t *counts, int32_t *starts,
                          int32_t *perm) {
    int64_t nb[3] = {1, 1, 1};
    for (int i = 0; i < dim; i++) nb[i] = (n[i] + m[i] - 1) / m[i];
    int64_t nbins = nb[0] * nb[1] * nb[2];
    for (int64_t b = 0; b < nbins; b++) counts[b] = 0;
    for (int64_t j = 0; j < M; j++) {
        int64_t c1 = bin_index(x[j], n[0], w);
        int64_t c2 = dim >= 2 ? bin_index(y[j], n[1], w) : 0;
        int64_t c3 = dim == 3 ? bin_index(z[j], n[2], w) : 0;
        int64_t b1 = c1 / m[0], b2 = dim >= 2 ? c2 / m[1] : 0, b3 = dim == 3 ? c3 / m[2] : 0;
        int64_t b = b1 + nb[0] * (b2 + nb[1] * b3);
        bin_of[j] = (int32_t)b;
        counts[b]++;
    }
    int64_t run = 0;
    for (int64_t b = 0; b < nbins; b++) {
        starts[b] = (int32_t)run;
        run += counts[b];
    }
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nbins ? nbins : 1));
    for (int64_t b = 0; b < nbins; b++) fill[b] = starts[b];
    for (int64_t j = 0; j < M; j++) perm[fill[bin_of[j]]++] = (int32_t)j;
    free(fill);
    return nbins;
}

int64_t oracle_binsort(int dim, const int64_t *n, const int64_t *m, int64_t M,
                       const double *x, const double *y, const double *z,
                       int32_t *bin_of, int32_t *counts, int32_t *starts,
                       int32_t *perm) {
    return binsort_by(dim, n, m, 0, M, x, y, z, bin_of, counts, starts, perm);
}

/* The same with points binned by window origin (bin_index with w > 0). */
int64_t oracle_binsort_origin(int dim, const int64_t *n, const int64_t *m, int w, int64_t M,
                              const double *x, const double *y, const double *z,
                              int32_t *bin_of, int32_t *counts, int32_t *starts,
                              int32_t *perm) {
    return binsort_by(dim, n, m, w, M, x, y, z, bin_of, counts, starts, perm);
}

/*
 * [cuFINUFFT] Sec. III-A SM step 1: each bin's points (a contiguous run of
 * perm) are cut into subproblems of at most msub points, bin by bin in bin
 * order.  Writes (bin, first sorted slot, point count) triples into `table`
 * when it is non-NULL and returns the number of subproblems.
 */
int64_t oracle_subproblems(int64_t nbins, const int32_t *counts,
                           const int32_t *starts, int64_t msub,
                           int32_t *table) {
    int64_t ns = 0;
    for (int64_t b = 0; b < nbins; b++) {
        for (int64_t off = 0; off < counts[b]; off += msub) {
            if (table) {
                int64_t left = counts[b] - off;
                table[3 * ns + 0] = (int32_t)b;
                table[3 * ns + 1] = (int32_t)(starts[b] + off);
                table[3 * ns + 2] = (int32_t)(left < msub ? left : msub);
            }
            ns++;
        }
    }
    return ns;
}

/* ---------------------------------------------------------------------- */
/* Quadrature                                                              */
/* ---------------------------------------------------------------------- */

/*
 * Gauss-Legendre nodes and weights on [-1, 1] (q >= 2 points): Newton
 * iteration on the Legendre three-term recurrence, started from the usual
 * cosine guesses.
 */
static void legendre(int q, double t, double *pq, double *pq1) {
    double p0 = 1.0, p1 = t;
    for (int k = 2; k <= q; k++) {
        double p2 = ((2.0 * k - 1.0) * t * p1 - (k - 1.0) * p0) / k;
        p0 = p1;
        p1 = p2;
    }
    *pq = p1;  /* P_q(t) */
    *pq1 = p0; /* P_{q-1}(t) */
}

void oracle_gauss_legendre(int q, double *nodes, double *weights) {
    for (int i = 0; i < q; i++) {
        double t = cos(ORACLE_PI * (i + 0.75) / (q + 0.5));
        double pq, pq1, dp;
        for (int it = 0; it < 100; it++) {
            legendre(q, t, &pq, &pq1);
            dp = q * (t * pq - pq1) / (t * t - 1.0);
            double dt = pq / dp;
            t -= dt;
            if (fabs(dt) < 1e-16) break;
        }
        legendre(q, t, &pq, &pq1);
        dp = q * (t * pq - pq1) / (t * t - 1.0);
        nodes[i] = t;
        weights[i] = 2.0 / ((1.0 - t * t) * dp * dp);
    }
}
