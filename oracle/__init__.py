"""Oracle for the 2D/3D type 1 / type 2 nonuniform FFT (double precision, CPU).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``nonuniform_fft_gb300``) never imports, links or runs it, and this package
imports nothing from the product library: the two share no code.

Source: "cuFINUFFT: a load-balanced GPU library for general-purpose nonuniform
FFTs" (Shih, Wright, Anden, Blaschke, Barnett), cited as [cuFINUFFT] with that
paper's section and equation numbers; and the GitHub finufft discussion #809
"CUFINUFFT binsize and performance", cited as [finufft#809].

Two oracles:

* **O1** -- the direct sums that *define* the transforms ([cuFINUFFT] Sec. I,
  eq. (1) type 1 and eq. (3) type 2), in double precision with compensated
  summation (``direct_type1`` / ``direct_type2``).
* **O2** -- the three-step NUFFT of [cuFINUFFT] Sec. II, step by step in the
  paper's order: spreading (eq. (7)-(8)), plain FFT (eq. (9)), truncation and
  correction (eq. (10)) for type 1; pre-correction and zero padding (eq. (11)),
  plain inverse FFT (eq. (12)), interpolation (Sec. II-B c) for type 2
  (``nufft_type1`` / ``nufft_type2``).  The spreading / interpolation loops
  and the direct sums are plain C (``nufft_oracle.c``); the FFT is numpy's.

Readings of points the paper leaves open (each also listed in the design notes):

* beta = 2.30 w.  Eq. (6) prints the factor with its digits lost; 2.30 is the
  value of the ES-kernel papers [cuFINUFFT] cites for sigma = 2, and the
  error-versus-tolerance pins check it.
* w = ceil(log10(1/eps)) + 1 (eq. (6)); a tolerance within 1e-9 (in log10) of a
  power of ten counts as that power, so decimal literals such as 1e-6 give the
  widths [finufft#809] lists (1e-3 -> 4, 1e-6 -> 7, 1e-9 -> 10, 1e-12 -> 13).
* Fine grid n_i: the smallest 2^a 3^b 5^c that is >= max(sigma N_i, 2 w)
  (Sec. II, text after eq. (6)); sigma = 2 unless a smaller upsampling factor
  is asked for.
* sigma < 2 ([cuFINUFFT] Sec. I-B limitation 3 and Sec. V name it as future
  work, citing the ES-kernel paper, but give no width rule for it): eq. (6)
  with its sigma dependence taken from the ES kernel's error law, which decays
  like exp(-pi w sqrt(1 - 1/sigma)).  Relative to sigma = 2 that stretches the
  digit count by 1/sqrt(2 (1 - 1/sigma)), and beta scales with
  (1 - 1/(2 sigma)) as in that paper:
      w = ceil(log10(1/eps) / sqrt(2 (1 - 1/sigma))) + 1,
      beta = 2.30 w (4/3) (1 - 1/(2 sigma)),
  which is eq. (6) itself at sigma = 2 (used verbatim there).  Accepted:
  1 < sigma <= 2.
* Fine-grid node l sits at l h (eq. (7)); a coordinate is reduced to one period
  [0, 2 pi) before use, so any finite coordinate is valid.
* A point touches the w nodes with kernel argument z in [-1, 1).
* phi-hat(xi) = 2 int_0^1 phi(z) cos(xi z) dz (eq. (4) with phi even) is
  computed by Gauss-Legendre quadrature after the substitution z = sin(theta),
  which makes the integrand smooth on [0, pi/2].
* Mode order: k1 fastest, each k_i increasing over I_N = [-floor(N/2), ...)
  (eq. (2)); mode k lives at fine-grid index k mod n.
* iflag: the sign of the exponent of both types; the FFT direction follows it.
  No normalisation anywhere (eq. (1), (3)).
"""
from __future__ import annotations

import ctypes
import fcntl
import math
import os
import platform
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nufft_oracle.c")
_LIB_PATH = os.path.join(_HERE, f"liboracle_{platform.machine()}.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C part of the oracle (gcc, no FMA contraction)."""
    lock_path = _LIB_PATH + ".lock"
    with open(lock_path, "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        fresh = (os.path.exists(_LIB_PATH)
                 and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
        if force or not fresh:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off",
                   "-fno-fast-math", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_direct_type1.argtypes = [I, I64, P, P, P, P, I, I64, P, I64, P, I64, P, P]
    lib.oracle_direct_type1.restype = None
    lib.oracle_direct_type2.argtypes = [I, P, P, P, P, P, I, I64, P, P]
    lib.oracle_direct_type2.restype = None
    lib.oracle_grid_coord.argtypes = [D, I64]
    lib.oracle_grid_coord.restype = D
    lib.oracle_spread.argtypes = [I, P, I, D, I64, P, P, P, P, P]
    lib.oracle_spread.restype = None
    lib.oracle_interp.argtypes = [I, P, I, D, I64, P, P, P, P, P]
    lib.oracle_interp.restype = None
    lib.oracle_binsort.argtypes = [I, P, P, I64, P, P, P, P, P, P, P]
    lib.oracle_binsort.restype = I64
    lib.oracle_binsort_origin.argtypes = [I, P, P, I, I64, P, P, P, P, P, P, P]
    lib.oracle_binsort_origin.restype = I64
    lib.oracle_subproblems.argtypes = [I64, P, P, I64, P]
    lib.oracle_subproblems.restype = I64
    lib.oracle_gauss_legendre.argtypes = [I, P, P]
    lib.oracle_gauss_legendre.restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def cpu_threads() -> int:
    """Host threads the oracle uses by default: every core this process may
    run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _thread_count(units: int, min_per_thread: int, threads: int | None, cap: int = 1 << 30) -> int:
    n = threads if threads else min(cpu_threads(), max(1, units // max(1, min_per_thread)))
    return max(1, min(n, cap, max(1, units)))


def _run_all(nthreads: int, fn):
    """fn(0), ..., fn(nthreads - 1), on separate threads when nthreads > 1
    (the C loops release the GIL while they run)."""
    if nthreads == 1:
        fn(0)
        return
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(nthreads) as ex:
        list(ex.map(fn, range(nthreads)))


def _on_threads(units: int, min_per_thread: int, threads: int | None, fn):
    """fn(lo, hi) over contiguous chunks of range(units), one per thread."""
    nthreads = _thread_count(units, min_per_thread, threads)
    bounds = np.linspace(0, units, nthreads + 1).astype(np.int64)

    def run(i):
        lo, hi = int(bounds[i]), int(bounds[i + 1])
        if hi > lo:
            fn(lo, hi)

    _run_all(nthreads, run)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.float64)


def _c128(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.complex128)


def _coords(pts):
    """(x[, y[, z]]) -> (dim, x, y-or-None, z-or-None) as contiguous float64
    arrays (float32 inputs are converted exactly)."""
    pts = [_f64(p) for p in pts]
    dim = len(pts)
    if dim not in (1, 2, 3):
        raise ValueError("dim must be 1, 2 or 3")
    return dim, pts[0], (pts[1] if dim >= 2 else None), (pts[2] if dim == 3 else None)


# --------------------------------------------------------------------------
# Parameters ([cuFINUFFT] Sec. II eq. (6) and the text after it)
# --------------------------------------------------------------------------

def _snap(v: float) -> float:
    """A value within 1e-9 (relative) of an integer counts as that integer, so
    decimal inputs do not flip a ceiling on rounding noise."""
    r = round(v)
    return float(r) if abs(v - r) <= 1e-9 * max(1.0, abs(v)) else v


def es_params(eps: float, sigma: float = 2.0) -> tuple[int, float]:
    """Kernel width w and ES shape beta for tolerance eps, [cuFINUFFT] eq. (6)
    at sigma = 2; the sigma < 2 reading in the module notes otherwise."""
    if not eps > 0:
        raise ValueError("eps must be > 0")
    if not 1.0 < sigma <= 2.0:
        raise ValueError("sigma must be in (1, 2]")
    L = _snap(-math.log10(eps))
    if sigma == 2.0:
        w = int(math.ceil(L)) + 1
        return w, 2.30 * w
    w = int(math.ceil(_snap(L / math.sqrt(2.0 * (1.0 - 1.0 / sigma))))) + 1
    return w, 2.30 * w * (4.0 / 3.0) * (1.0 - 0.5 / sigma)


def fine_grid_size(N: int, w: int, sigma: float = 2.0) -> int:
    """Smallest 2^a 3^b 5^c >= max(sigma N, 2 w)."""
    target = max(int(math.ceil(_snap(sigma * N))), 2 * w)
    n = target
    while True:
        m = n
        for p in (2, 3, 5):
            while m % p == 0:
                m //= p
        if m == 1:
            return n
        n += 1


def es_kernel(z, beta: float):
    """phi_beta(z) of [cuFINUFFT] eq. (5)."""
    z = np.asarray(z, dtype=np.float64)
    out = np.zeros_like(z)
    inside = np.abs(z) <= 1.0
    out[inside] = np.exp(beta * (np.sqrt(1.0 - z[inside] ** 2) - 1.0))
    return out


def gauss_legendre(q: int) -> tuple[np.ndarray, np.ndarray]:
    nodes = np.zeros(q)
    weights = np.zeros(q)
    _load().oracle_gauss_legendre(q, _ptr(nodes), _ptr(weights))
    return nodes, weights


def phihat(xi, beta: float, q: int = 200):
    """Fourier transform of the ES kernel under eq. (4):
    phi-hat(xi) = int_{-1}^{1} phi(z) e^{-i xi z} dz = 2 int_0^1 phi(z) cos(xi z) dz,
    evaluated with z = sin(theta) as 2 int_0^{pi/2} e^{beta(cos theta - 1)}
    cos(xi sin theta) cos theta dtheta by q-point Gauss-Legendre."""
    t, wt = gauss_legendre(q)
    theta = (t + 1.0) * (math.pi / 4.0)
    dtheta = wt * (math.pi / 4.0)
    xi = np.asarray(xi, dtype=np.float64)
    integrand = (np.exp(beta * (np.cos(theta) - 1.0)) * np.cos(theta))
    return 2.0 * np.cos(np.multiply.outer(xi, np.sin(theta))) @ (integrand * dtheta)


def mode_indices(N: int) -> np.ndarray:
    """I_N of [cuFINUFFT] eq. (2), increasing."""
    return np.arange(-(N // 2), N - N // 2, dtype=np.int64)


def correction_factors(N: int, n: int, w: int, beta: float) -> np.ndarray:
    """Per-dimension correction p(k) = (2/w) / phi-hat(alpha k), alpha = w pi / n,
    for k in I_N ([cuFINUFFT] text after eq. (10))."""
    alpha = w * math.pi / n
    return (2.0 / w) / phihat(alpha * mode_indices(N), beta)


# --------------------------------------------------------------------------
# O1: direct sums
# --------------------------------------------------------------------------

def direct_type1(pts, c, N, iflag: int, modes=None, threads: int | None = None) -> np.ndarray:
    """f_k = sum_j c_j exp(+-i k.x_j) ([cuFINUFFT] eq. (1)).

    modes=None: every mode of I_N1 x I_N2 (x I_N3), shaped (N3,) N2, N1.
    Otherwise ``modes`` is a list of per-dimension integer lists (K1, K2[, K3])
    and the result is the tensor grid of those modes, shaped (K3,) K2, K1.
    The points are cut into chunks summed on separate threads (the C loop
    releases the GIL); the chunk sums are added in double."""
    dim, x, y, z = _coords(pts)
    c = _c128(c)
    if modes is None:
        modes = [mode_indices(n) for n in N]
    ks = [np.ascontiguousarray(np.asarray(k, dtype=np.int64)) for k in modes]
    if len(ks) != dim:
        raise ValueError("one mode list per dimension")
    k2 = ks[1] if dim >= 2 else np.zeros(1, np.int64)
    k3 = ks[2] if dim == 3 else np.zeros(1, np.int64)
    shape = tuple(len(k) for k in reversed(ks))
    total = int(np.prod(shape))
    M = x.size
    nthreads = _thread_count(M, 20000, threads)
    bounds = np.linspace(0, M, nthreads + 1).astype(np.int64)
    parts = [np.zeros(total, dtype=np.complex128) for _ in range(nthreads)]
    lib = _load()

    def run(i):
        lo, hi = int(bounds[i]), int(bounds[i + 1])
        if hi <= lo:
            return
        yy = None if y is None else y[lo:]
        zz = None if z is None else z[lo:]
        lib.oracle_direct_type1(dim, hi - lo, _ptr(x[lo:]), _ptr(yy), _ptr(zz),
                                _ptr(c[lo:]), int(iflag), ks[0].size, _ptr(ks[0]),
                                k2.size, _ptr(k2), k3.size, _ptr(k3),
                                _ptr(parts[i]))

    if nthreads == 1:
        run(0)
    else:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(run, range(nthreads)))
    out = parts[0]
    for p in parts[1:]:
        out = out + p
    return out.reshape(shape)


def direct_type2(pts, f, N, iflag: int, targets=None, threads: int | None = None) -> np.ndarray:
    """c_j = sum_k f_k exp(+-i k.x_j) ([cuFINUFFT] eq. (3)) at the listed
    targets (user indices; all points when None).  The targets are cut into
    chunks evaluated on separate threads; each target's sum is independent."""
    dim, x, y, z = _coords(pts)
    f = _c128(f).ravel()
    Nn = np.asarray(list(N), dtype=np.int64)
    if f.size != int(np.prod(Nn)):
        raise ValueError("f has the wrong number of modes")
    t = np.arange(x.size, dtype=np.int64) if targets is None else \
        np.ascontiguousarray(np.asarray(targets, dtype=np.int64))
    out = np.zeros(t.size, dtype=np.complex128)
    lib = _load()

    def run(lo, hi):
        lib.oracle_direct_type2(dim, _ptr(Nn), _ptr(x), _ptr(y), _ptr(z), _ptr(f),
                                int(iflag), hi - lo, _ptr(t[lo:]), _ptr(out[lo:]))

    _on_threads(t.size, max(1, (1 << 22) // max(1, f.size)), threads, run)
    return out


# --------------------------------------------------------------------------
# O2: three-step NUFFT ([cuFINUFFT] Sec. II)
# --------------------------------------------------------------------------

def plan_params(N, eps: float, sigma: float = 2.0):
    w, beta = es_params(eps, sigma)
    n = [fine_grid_size(Ni, w, sigma) for Ni in N]
    return w, beta, n


def spread(pts, c, n, w: int, beta: float, threads: int | None = None) -> np.ndarray:
    """Type 1 step 1, eq. (7): fine grid b shaped (n3,) n2, n1 (x fastest).

    b is a sum over points, so the points are cut into contiguous chunks in
    user order, each chunk spread by the plain C loop into its own fine grid
    on its own thread, and the chunk grids are added in double (rounding
    order differs from one serial loop only in where the partial sums meet).
    The thread count is capped so the chunk grids take at most about 4 GB."""
    dim, x, y, z = _coords(pts)
    c = _c128(c)
    nn = np.asarray(list(n), dtype=np.int64)
    shape = tuple(reversed(list(n)))
    grid_bytes = 16 * int(np.prod(shape))
    cap = max(1, (4 << 30) // max(1, grid_bytes))
    nthreads = _thread_count(x.size, 20000, threads, cap)
    grids = [np.empty(shape, dtype=np.complex128) for _ in range(nthreads)]
    bounds = np.linspace(0, x.size, nthreads + 1).astype(np.int64)
    lib = _load()

    def run(i):
        lo, hi = int(bounds[i]), int(bounds[i + 1])
        lib.oracle_spread(dim, _ptr(nn), w, beta, hi - lo, _ptr(x[lo:]),
                          None if y is None else _ptr(y[lo:]),
                          None if z is None else _ptr(z[lo:]), _ptr(c[lo:]), _ptr(grids[i]))

    _run_all(nthreads, run)
    b = grids[0]
    for g in grids[1:]:
        b += g
    return b


def interp(pts, b, n, w: int, beta: float, threads: int | None = None) -> np.ndarray:
    """Type 2 step 3 (Sec. II-B c): c_j = sum_l b_l psi_per(l h - x_j).
    Each c_j is independent, so contiguous chunks of points run on separate
    threads of the plain C loop."""
    dim, x, y, z = _coords(pts)
    b = _c128(b)
    nn = np.asarray(list(n), dtype=np.int64)
    c = np.zeros(x.size, dtype=np.complex128)
    lib = _load()

    def run(lo, hi):
        lib.oracle_interp(dim, _ptr(nn), w, beta, hi - lo, _ptr(x[lo:]),
                          None if y is None else _ptr(y[lo:]),
                          None if z is None else _ptr(z[lo:]), _ptr(b), _ptr(c[lo:]))

    _on_threads(x.size, 20000, threads, run)
    return c


def _fft(b: np.ndarray, iflag: int) -> np.ndarray:
    """Unnormalised FFT over every axis with exponent sign sign(iflag)
    (eq. (9) for iflag < 0, eq. (12) for iflag >= 0)."""
    if iflag < 0:
        return np.fft.fftn(b)
    return np.fft.ifftn(b, norm="forward")


def _fine_index(N: int, n: int) -> np.ndarray:
    return np.mod(mode_indices(N), n)


def _outer(ps):
    """Tensor product p1(k1) p2(k2) [p3(k3)] shaped like f: (N3,) N2, N1."""
    out = ps[0]
    for p in ps[1:]:
        out = np.multiply.outer(p, out)
    return out


def nufft_type1(pts, c, N, eps: float, iflag: int, sigma: float = 2.0,
                threads: int | None = None) -> np.ndarray:
    """O2 type 1: spread (eq. (7)), FFT (eq. (9)), truncate + correct (eq. (10)).
    Returns f shaped (N3,) N2, N1."""
    N = list(N)
    w, beta, n = plan_params(N, eps, sigma)
    b = spread(pts, c, n, w, beta, threads)
    bhat = _fft(b, iflag)
    idx = [_fine_index(Ni, ni) for Ni, ni in zip(N, n)]
    sub = bhat[np.ix_(*reversed(idx))]
    p = _outer([correction_factors(Ni, ni, w, beta) for Ni, ni in zip(N, n)])
    return p * sub


def nufft_type2(pts, f, N, eps: float, iflag: int, sigma: float = 2.0,
                threads: int | None = None) -> np.ndarray:
    """O2 type 2: pre-correct + zero-pad (eq. (11)), FFT (eq. (12)),
    interpolate (Sec. II-B c).  f shaped (N3,) N2, N1 or flat."""
    N = list(N)
    w, beta, n = plan_params(N, eps, sigma)
    f = _c128(f).reshape(tuple(reversed(N)))
    p = _outer([correction_factors(Ni, ni, w, beta) for Ni, ni in zip(N, n)])
    bhat = np.zeros(tuple(reversed(n)), dtype=np.complex128)
    idx = [_fine_index(Ni, ni) for Ni, ni in zip(N, n)]
    bhat[np.ix_(*reversed(idx))] = p * f
    b = _fft(bhat, iflag)
    return interp(pts, b, n, w, beta, threads)


# --------------------------------------------------------------------------
# Integer setpts results ([cuFINUFFT] Sec. III-A)
# --------------------------------------------------------------------------

def grid_coord(x: float, n: int) -> float:
    """Fine-grid coordinate g in [0, n) of one coordinate (eq. (7) geometry)."""
    return _load().oracle_grid_coord(float(x), int(n))


def binsort(pts, n, m, msub: int, origin_w: int = 0):
    """Bin of each point, bin counts, bin starts, the stable permutation t and
    the subproblem table (bin, first sorted slot, count) rows.

    origin_w = 0: a point's bin is the bin of its cell floor(g) ([cuFINUFFT]
    Sec. III-A).  origin_w = w > 0: the bin of its window origin shifted by
    floor(w/2), (ceil(g - w/2) + floor(w/2)) mod n, with ceil(g - w/2) the
    first of the w nodes the point touches (Sec. II-B)."""
    dim, x, y, z = _coords(pts)
    nn = np.asarray(list(n), dtype=np.int64)
    mm = np.asarray(list(m), dtype=np.int64)
    nb = [-(-int(a) // int(b)) for a, b in zip(nn, mm)]
    nbins = int(np.prod(nb))
    bin_of = np.zeros(x.size, np.int32)
    counts = np.zeros(nbins, np.int32)
    starts = np.zeros(nbins, np.int32)
    perm = np.zeros(x.size, np.int32)
    lib = _load()
    if origin_w:
        lib.oracle_binsort_origin(dim, _ptr(nn), _ptr(mm), int(origin_w), x.size, _ptr(x), _ptr(y),
                                  _ptr(z), _ptr(bin_of), _ptr(counts), _ptr(starts), _ptr(perm))
    else:
        lib.oracle_binsort(dim, _ptr(nn), _ptr(mm), x.size, _ptr(x), _ptr(y), _ptr(z),
                           _ptr(bin_of), _ptr(counts), _ptr(starts), _ptr(perm))
    nsub = lib.oracle_subproblems(nbins, _ptr(counts), _ptr(starts), int(msub), None)
    table = np.zeros((nsub, 3), np.int32)
    lib.oracle_subproblems(nbins, _ptr(counts), _ptr(starts), int(msub), _ptr(table))
    return {"bin_of": bin_of, "counts": counts, "starts": starts, "perm": perm,
            "subproblems": table}


def rel_l2(a, b) -> float:
    """||a - b||_2 / ||b||_2, the error measure of [cuFINUFFT] Sec. IV-C."""
    a = np.asarray(a).ravel()
    b = np.asarray(b).ravel()
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))
