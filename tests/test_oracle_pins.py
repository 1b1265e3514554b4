"""Pins of the CPU oracle against facts fixed by the paper and by mathematics.

Nothing here compares the oracle with itself: each check is a value printed
on the pages (golden fixture), a closed form, an identity that any correct
transform obeys, a special case that reduces to a library FFT, or the accuracy
bound the method claims.  Sources: "cuFINUFFT: a load-balanced GPU library for
general-purpose nonuniform FFTs" ([cuFINUFFT], section / equation numbers are
that paper's) and the GitHub finufft discussion #809 "CUFINUFFT binsize and
performance" ([finufft#809]).
"""
import math
import os
import warnings

import numpy as np
import pytest
from scipy import integrate

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


def _rand_pts(dim, M, rng=RNG):
    return [rng.uniform(-np.pi, np.pi, M) for _ in range(dim)]


def _rand_c(M, rng=RNG):
    return rng.standard_normal(M) + 1j * rng.standard_normal(M)


# ---------------------------------------------------------------- parameters

def test_width_table_golden():
    """[finufft#809] 'Tolerance (Kernel Width ns)': 1e-3->4, 1e-6->7, 1e-9->10, 1e-12->13."""
    rows = [l.split() for l in open(os.path.join(GOLDEN, "es_width_table.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 4
    for tol, width in rows:
        w, beta = oracle.es_params(float(tol))
        assert w == int(width)
        assert beta == pytest.approx(2.30 * w)


def test_width_rule_between_powers():
    # eq. (6): w = ceil(log10(1/eps)) + 1
    assert oracle.es_params(5e-4)[0] == 5     # log10(2000) = 3.3 -> 4 -> w = 5
    assert oracle.es_params(1e-5)[0] == 6
    assert oracle.es_params(0.5)[0] == 2      # log10(2) = 0.3 -> 1 -> 2
    assert oracle.es_params(1e-2)[0] == 3


@pytest.mark.parametrize("N,w,n", [(64, 6, 128), (1024, 6, 2048), (128, 7, 256),
                                   (64, 13, 128), (7, 6, 15), (4, 13, 27), (11, 6, 24),
                                   (100, 6, 200), (1, 2, 4), (3, 2, 6)])
def test_fine_grid_size(N, w, n):
    # smallest 2^a 3^b 5^c >= max(2N, 2w), worked by hand
    assert oracle.fine_grid_size(N, w) == n


def test_gauss_legendre_exact_on_polynomials():
    # a q-point Gauss rule integrates x^k exactly on [-1,1] for k <= 2q-1
    for q in (2, 5, 16, 200):
        t, wt = oracle.gauss_legendre(q)
        assert np.all(np.diff(np.sort(t)) > 0) and np.all(np.abs(t) < 1)
        for k in range(0, min(2 * q, 40)):
            exact = 0.0 if k % 2 else 2.0 / (k + 1)
            assert np.dot(wt, t ** k) == pytest.approx(exact, abs=1e-14)


def test_phihat_beta0_closed_form():
    # beta = 0: phi = 1 on [-1,1], so phi-hat(xi) = 2 sin(xi)/xi (eq. (4))
    xi = np.array([1e-3, 0.5, 1.0, 3.0, 7.5, 10.0])
    assert np.allclose(oracle.phihat(xi, 0.0), 2 * np.sin(xi) / xi, rtol=1e-14, atol=0)


@pytest.mark.parametrize("w", [2, 3, 6, 7, 13, 16])
def test_phihat_against_adaptive_quadrature(w):
    """phi-hat of eq. (4) for the ES kernel (eq. (5)), checked against scipy's
    adaptive quadrature of the untransformed integral over z."""
    beta = 2.30 * w
    xis = np.linspace(0.0, w * np.pi / 4 * 1.01, 7)
    got = oracle.phihat(xis, beta)
    for xi, g in zip(xis, got):
        f = lambda z: math.exp(beta * (math.sqrt(max(0.0, 1 - z * z)) - 1)) * math.cos(xi * z)
        with warnings.catch_warnings():
            warnings.simplefilter("ignore", integrate.IntegrationWarning)
            ref, _ = integrate.quad(f, -1.0, 1.0, epsabs=1e-15, epsrel=1e-14, limit=400)
        assert g == pytest.approx(ref, rel=2e-13)


def test_es_kernel_values():
    # eq. (5): phi(0) = 1, phi(+-1) = e^{-beta}, zero outside [-1,1]
    beta = 13.8
    v = oracle.es_kernel([0.0, 1.0, -1.0, 1.0000001, -3.0], beta)
    assert v[0] == 1.0
    assert v[1] == pytest.approx(math.exp(-beta), rel=1e-15)
    assert v[2] == pytest.approx(math.exp(-beta), rel=1e-15)
    assert v[3] == 0.0 and v[4] == 0.0


# ---------------------------------------------------------------- O1: direct sums

@pytest.mark.parametrize("N", [(9,), (5, 8), (6, 4, 7)])
@pytest.mark.parametrize("iflag", [-1, 1])
def test_direct_type1_single_point(N, iflag):
    """c = 1 at one point: f_k = exp(s i k.x) exactly (eq. (1)); at x = 0, f == 1."""
    dim = len(N)
    x0 = RNG.uniform(-np.pi, np.pi, dim)
    f = oracle.direct_type1([[v] for v in x0], [1.0], N, iflag)
    ks = np.meshgrid(*[oracle.mode_indices(n) for n in reversed(N)], indexing="ij")
    phase = sum(k * xv for k, xv in zip(reversed(ks), x0))
    assert f.shape == tuple(reversed(N))
    assert np.allclose(f, np.exp(np.sign(iflag) * 1j * phase), rtol=0, atol=1e-14)
    f0 = oracle.direct_type1([[0.0]] * dim, [1.0], N, iflag)
    assert np.allclose(f0, 1.0, atol=1e-15)


@pytest.mark.parametrize("N", [(9,), (5, 8), (6, 4, 7)])
@pytest.mark.parametrize("iflag", [-1, 1])
def test_direct_type2_single_mode(N, iflag):
    """f = delta at mode k0: c_j = exp(s i k0.x_j) (eq. (3))."""
    dim = len(N)
    pts = _rand_pts(dim, 13)
    k0 = [oracle.mode_indices(n)[RNG.integers(n)] for n in N]
    f = np.zeros(tuple(reversed(N)), complex)
    f[tuple(k + n // 2 for k, n in zip(reversed(k0), reversed(N)))] = 1.0
    c = oracle.direct_type2(pts, f, N, iflag)
    phase = sum(k * p for k, p in zip(k0, pts))
    assert np.allclose(c, np.exp(np.sign(iflag) * 1j * phase), rtol=0, atol=1e-13)


@pytest.mark.parametrize("N", [(10,), (6, 10), (4, 6, 5)])
@pytest.mark.parametrize("iflag", [-1, 1])
def test_direct_equispaced_is_numpy_fft(N, iflag):
    """Points on the N1 x N2 (x N3) lattice x_a = 2 pi a / N: type 1 is the
    plain DFT of the strengths, i.e. numpy's FFT (sign s) read at k mod N.
    Coordinates >= pi are moved down by 2 pi (the sums are 2 pi periodic)."""
    dim = len(N)
    grids = np.meshgrid(*[2 * np.pi * np.arange(n) / n for n in reversed(N)], indexing="ij")
    coords = [g.ravel() for g in reversed(grids)]
    coords = [np.where(cc >= np.pi, cc - 2 * np.pi, cc) for cc in coords]
    c = _rand_c(int(np.prod(N))).reshape(tuple(reversed(N)))
    f = oracle.direct_type1(coords, c.ravel(), N, iflag)
    F = np.fft.fftn(c) if iflag < 0 else np.fft.ifftn(c) * c.size
    idx = [np.mod(oracle.mode_indices(n), n) for n in reversed(N)]
    assert np.allclose(f, F[np.ix_(*idx)], rtol=0, atol=1e-11)
    # type 2 at the lattice points is the DFT of the opposite sign
    fk = _rand_c(c.size).reshape(c.shape)
    c2 = oracle.direct_type2(coords, fk, N, iflag)
    G = np.zeros(c.shape, complex)
    G[np.ix_(*idx)] = fk
    ref = np.fft.ifftn(G) * G.size if iflag >= 0 else np.fft.fftn(G)
    assert np.allclose(c2, ref.ravel(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("N", [(11,), (7, 6), (4, 5, 6)])
def test_direct_adjoint_identity(N):
    """<T1_s(c), f> = <c, T2_{-s}(f)>: type 2 is the adjoint of type 1 (Sec. I)."""
    dim = len(N)
    pts = _rand_pts(dim, 40)
    c = _rand_c(40)
    f = _rand_c(int(np.prod(N)))
    for s in (-1, 1):
        lhs = np.vdot(oracle.direct_type1(pts, c, N, s).ravel(), f)
        rhs = np.vdot(c, oracle.direct_type2(pts, f, N, -s))
        assert lhs == pytest.approx(rhs, rel=1e-13)


def test_direct_shift_and_period():
    """x -> x + d multiplies f_k by exp(s i k d); x -> x + 2 pi changes nothing."""
    N = (6, 8)
    pts = _rand_pts(2, 30)
    c = _rand_c(30)
    f = oracle.direct_type1(pts, c, N, -1)
    d = 0.37
    g = oracle.direct_type1([pts[0] + d, pts[1]], c, N, -1)
    k1 = oracle.mode_indices(6)[None, :]
    assert np.allclose(g, f * np.exp(-1j * k1 * d), atol=1e-12)
    h = oracle.direct_type1([pts[0] + 2 * np.pi, pts[1] - 4 * np.pi], c, N, -1)
    assert np.allclose(h, f, atol=1e-11)


def test_direct_type1_mode_subset_matches_full():
    N = (10, 12)
    pts = _rand_pts(2, 50)
    c = _rand_c(50)
    full = oracle.direct_type1(pts, c, N, 1)
    k1 = np.array([-5, 0, 4])
    k2 = np.array([-6, 5])
    sub = oracle.direct_type1(pts, c, N, 1, modes=[k1, k2])
    assert np.allclose(sub, full[np.ix_(k2 + 6, k1 + 5)], rtol=0, atol=1e-13)
    # threaded chunking gives the same sums
    thr = oracle.direct_type1(pts, c, N, 1, threads=4)
    assert np.allclose(thr, full, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- O2: NUFFT

@pytest.mark.parametrize("dim,N,M", [(1, (48,), 3000), (2, (40, 32), 3000), (3, (16, 12, 20), 3000)])
@pytest.mark.parametrize("eps", [1e-2, 1e-3, 1e-5, 1e-6, 1e-9, 1e-12])
def test_nufft_error_close_to_eps(dim, N, M, eps):
    """[cuFINUFFT] Sec. II: with w, beta from eq. (6) the relative l2 error is
    'close to eps'.  Both types, both signs, against the direct sums.  The
    paper gives no hard bound; 'close' is taken as within [eps/4, 4 eps].  The
    error is a few times the kernel's edge value e^-beta = 10^-w, so a width off
    by one in either direction moves it by about ten and fails the check."""
    rng = np.random.default_rng(7)
    pts = [rng.uniform(-np.pi, np.pi, M) for _ in range(dim)]
    c = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    f = rng.standard_normal(int(np.prod(N))) + 1j * rng.standard_normal(int(np.prod(N)))
    for iflag in (-1, 1):
        e1 = oracle.rel_l2(oracle.nufft_type1(pts, c, N, eps, iflag),
                           oracle.direct_type1(pts, c, N, iflag))
        e2 = oracle.rel_l2(oracle.nufft_type2(pts, f, N, eps, iflag),
                           oracle.direct_type2(pts, f, N, iflag))
        assert e1 <= 4 * eps and e2 <= 4 * eps
        if eps >= 1e-11:          # below that, double rounding sets the floor
            assert e1 >= eps / 4 and e2 >= eps / 4


@pytest.mark.parametrize("dim,N,M", [(1, (48,), 3001), (2, (40, 32), 3001), (3, (16, 12, 20), 2003)])
@pytest.mark.parametrize("eps", [1e-6, 1e-12])
def test_nufft_threaded_chunks_close_to_eps(dim, N, M, eps):
    """The oracle spreads and interpolates contiguous chunks of points on
    separate threads (spread: one fine grid per chunk, summed).  With an odd
    point count split three ways, a chunk offset or a dropped partial grid
    would miss the direct sums by far more than eps; the threaded result must
    stay within [eps/4, 4 eps] of eq. (1) / (3) like the one-thread one."""
    rng = np.random.default_rng(8)
    pts = [rng.uniform(-np.pi, np.pi, M) for _ in range(dim)]
    c = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    f = rng.standard_normal(int(np.prod(N))) + 1j * rng.standard_normal(int(np.prod(N)))
    e1 = oracle.rel_l2(oracle.nufft_type1(pts, c, N, eps, -1, threads=3),
                       oracle.direct_type1(pts, c, N, -1))
    e2 = oracle.rel_l2(oracle.nufft_type2(pts, f, N, eps, 1, threads=3),
                       oracle.direct_type2(pts, f, N, 1, threads=3))
    assert e1 <= 4 * eps and e2 <= 4 * eps
    if eps >= 1e-11:
        assert e1 >= eps / 4 and e2 >= eps / 4


def test_sigma_rule_is_eq6_at_two():
    """The sigma < 2 reading reduces to eq. (6) itself at sigma = 2."""
    for tol in (0.5, 1e-2, 1e-3, 5e-4, 1e-5, 1e-6, 1e-9, 1e-12, 1e-15):
        assert oracle.es_params(tol, 2.0) == oracle.es_params(tol)
        for N in (1, 7, 64, 1000):
            w = oracle.es_params(tol)[0]
            assert oracle.fine_grid_size(N, w, 2.0) == oracle.fine_grid_size(N, w)


def test_sigma_rule_hand_values():
    """Worked by hand: sigma = 1.25, eps = 1e-6: 6 / sqrt(2 * 0.2) = 9.49 ->
    w = 11, beta = 2.30 * 11 * (4/3) * 0.6 = 20.24; sigma = 1.5, eps = 1e-3:
    3 / sqrt(2/3) = 3.67 -> w = 5, beta = 2.30 * 5 * (4/3) * (2/3) = 10.22;
    grids: 1.25 * 100 = 125 = 5^3; 1.5 * 64 = 96 = 2^5 3; 1.5 * 30 = 45 but
    2 w = 22 < 45 -> 45 = 3^2 5; 1.25 * 10 = 12.5 -> 13 -> 15 = 3 5."""
    w, beta = oracle.es_params(1e-6, 1.25)
    assert w == 11 and abs(beta - 20.24) < 1e-12
    w, beta = oracle.es_params(1e-3, 1.5)
    assert w == 5 and abs(beta - 2.30 * 5 * 8 / 9) < 1e-12
    assert oracle.fine_grid_size(100, 11, 1.25) == 125
    assert oracle.fine_grid_size(64, 5, 1.5) == 96
    assert oracle.fine_grid_size(30, 11, 1.5) == 45
    assert oracle.fine_grid_size(10, 4, 1.25) == 15
    with pytest.raises(ValueError):
        oracle.es_params(1e-6, 1.0)
    with pytest.raises(ValueError):
        oracle.es_params(1e-6, 2.5)


@pytest.mark.parametrize("dim,N,M", [(1, (200,), 3000), (2, (48, 40), 3000), (3, (24, 20, 28), 2000)])
@pytest.mark.parametrize("sigma", [1.25, 1.5])
@pytest.mark.parametrize("eps", [1e-2, 1e-3, 1e-6, 1e-9])
def test_nufft_error_close_to_eps_sigma(dim, N, M, sigma, eps):
    """sigma < 2 ([cuFINUFFT] Sec. I-B limitation 3): with the stretched
    eq. (6) the error against the direct sums stays 'close to eps', here
    within [eps/8, 3 eps] for both types and signs, on a grid smaller than
    the sigma = 2 one.  A grid or beta taken from sigma = 2 by mistake makes
    the error orders of magnitude smaller than eps; a beta for the wrong
    sigma, orders larger."""
    rng = np.random.default_rng(9)
    pts = [rng.uniform(-np.pi, np.pi, M) for _ in range(dim)]
    c = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    f = rng.standard_normal(int(np.prod(N))) + 1j * rng.standard_normal(int(np.prod(N)))
    w, _, n = oracle.plan_params(N, eps, sigma)
    assert any(ni < 2 * Ni for ni, Ni in zip(n, N))
    for iflag in (-1, 1):
        e1 = oracle.rel_l2(oracle.nufft_type1(pts, c, N, eps, iflag, sigma),
                           oracle.direct_type1(pts, c, N, iflag))
        e2 = oracle.rel_l2(oracle.nufft_type2(pts, f, N, eps, iflag, sigma),
                           oracle.direct_type2(pts, f, N, iflag))
        assert eps / 8 <= e1 <= 3 * eps and eps / 8 <= e2 <= 3 * eps, (e1 / eps, e2 / eps)


@pytest.mark.parametrize("N", [(20,), (16, 12), (8, 10, 6)])
def test_nufft_single_point(N):
    """c = 1 at x0: f_k ~ exp(-i k.x0) (|f_k| = 1) within eps; x0 anywhere,
    including the fold boundaries -pi and just below pi.  The error per mode
    peaks at the edge modes, where the correction factor is largest, so the
    bound here is 20 eps; it targets sign, origin and index mistakes, which
    give errors of order one.  The l2 accuracy itself is pinned by the sweep."""
    eps = 1e-9
    dim = len(N)
    for x0 in ([-np.pi] * dim, [np.pi * (1 - 1e-15)] * dim, list(RNG.uniform(-np.pi, np.pi, dim)),
               [0.0] * dim):
        f = oracle.nufft_type1([[v] for v in x0], [1.0], N, eps, -1)
        ks = np.meshgrid(*[oracle.mode_indices(n) for n in reversed(N)], indexing="ij")
        ref = np.exp(-1j * sum(k * v for k, v in zip(reversed(ks), x0)))
        assert oracle.rel_l2(f, ref) < 20 * eps


@pytest.mark.parametrize("N", [(20,), (16, 12), (8, 10, 6)])
def test_nufft_single_mode(N):
    """f = delta at k0: c_j ~ exp(+i k0.x_j) (eq. (3)), k0 the corner mode
    (-N1/2, -N2/2, ...), where the correction is largest: bound 20 eps."""
    eps = 1e-9
    dim = len(N)
    pts = _rand_pts(dim, 200)
    k0 = [oracle.mode_indices(n)[0] for n in N]      # the most negative mode: the edge
    f = np.zeros(tuple(reversed(N)), complex)
    f[(0,) * dim] = 1.0
    c = oracle.nufft_type2(pts, f, N, eps, 1)
    ref = np.exp(1j * sum(k * p for k, p in zip(k0, pts)))
    assert oracle.rel_l2(c, ref) < 20 * eps


@pytest.mark.parametrize("N", [(15,), (10, 14), (6, 8, 5)])
def test_nufft_adjoint_identity(N):
    """O2 type 1 (sign s) and O2 type 2 (sign -s) are exact transposes of each
    other: spreading/interpolation, FFT of opposite signs and the real diagonal
    correction.  Holds to rounding, at any eps."""
    dim = len(N)
    pts = _rand_pts(dim, 300)
    c = _rand_c(300)
    f = _rand_c(int(np.prod(N)))
    for eps in (1e-2, 1e-6):
        for s in (-1, 1):
            lhs = np.vdot(oracle.nufft_type1(pts, c, N, eps, s).ravel(), f)
            rhs = np.vdot(c, oracle.nufft_type2(pts, f, N, eps, -s))
            assert lhs == pytest.approx(rhs, rel=1e-12)


def test_nufft_linearity_and_conjugation():
    N = (12, 10)
    pts = _rand_pts(2, 100)
    c1, c2 = _rand_c(100), _rand_c(100)
    a, b = 0.3 - 1.1j, -2.0 + 0.5j
    lhs = oracle.nufft_type1(pts, a * c1 + b * c2, N, 1e-6, -1)
    rhs = a * oracle.nufft_type1(pts, c1, N, 1e-6, -1) + b * oracle.nufft_type1(pts, c2, N, 1e-6, -1)
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-11)
    r = RNG.standard_normal(100)
    assert np.allclose(oracle.nufft_type1(pts, r, N, 1e-6, 1),
                       np.conj(oracle.nufft_type1(pts, r, N, 1e-6, -1)), atol=1e-12)


def test_nufft_fold_invariance():
    """Shifting every coordinate by a multiple of 2 pi leaves the result unchanged
    (the fold to [0, 2 pi)), up to the rounding of the shifted coordinate."""
    N = (8, 6, 10)
    pts = _rand_pts(3, 60)
    c = _rand_c(60)
    f = oracle.nufft_type1(pts, c, N, 1e-9, -1)
    g = oracle.nufft_type1([pts[0] + 2 * np.pi, pts[1] - 2 * np.pi, pts[2] + 6 * np.pi],
                           c, N, 1e-9, -1)
    assert oracle.rel_l2(g, f) < 1e-12


# ---------------------------------------------------------------- bin sort

def test_grid_coord_landmarks():
    """Eq. (7): node l at l h, h = 2 pi / n, coordinates taken mod 2 pi."""
    n = 64
    h = 2 * np.pi / n
    assert oracle.grid_coord(0.0, n) == 0.0
    assert oracle.grid_coord(-np.pi, n) == 32.0
    assert oracle.grid_coord(np.pi, n) == 32.0
    assert oracle.grid_coord(2 * np.pi, n) == 0.0
    assert oracle.grid_coord(-1e-300, n) == 0.0            # rounds to 2 pi -> wraps to 0
    assert math.floor(oracle.grid_coord(-1e-9, n)) == 63
    assert math.floor(oracle.grid_coord(np.pi - 1e-12, n)) == 31
    assert oracle.grid_coord(3.5 * h, n) == pytest.approx(3.5, abs=1e-12)
    assert oracle.grid_coord(-3.5 * h, n) == pytest.approx(60.5, abs=1e-12)


def test_binsort_handpicked():
    """Bins of m1 x m2 cells, x fastest (Sec. III-A); edge bins smaller."""
    n = (20, 12)
    m = (8, 8)                       # bins: 3 x 2, the last column/row is smaller
    h1, h2 = 2 * np.pi / 20, 2 * np.pi / 12
    cells = [(0.5, 0.5), (19.5, 11.5), (8.5, 0.5), (16.2, 8.1), (7.9, 7.9), (0.5, 0.5)]
    x = [a * h1 for a, _ in cells]
    y = [b * h2 for _, b in cells]
    r = oracle.binsort([x, y], n, m, msub=2)
    # bin = (cell1 // 8) + 3 * (cell2 // 8)
    assert list(r["bin_of"]) == [0, 5, 1, 5, 0, 0]
    assert list(r["counts"]) == [3, 1, 0, 0, 0, 2]
    assert list(r["starts"]) == [0, 3, 4, 4, 4, 4]
    assert list(r["perm"]) == [0, 4, 5, 2, 1, 3]        # stable within a bin
    assert r["subproblems"].tolist() == [[0, 0, 2], [0, 2, 1], [1, 3, 1], [5, 4, 2]]


def test_binsort_by_window_origin_handpicked():
    """Binning by window origin: the bin index of a point at fine coordinate g
    is (ceil(g - w/2) + floor(w/2)) mod n -- for odd w the node nearest g
    (ties down), for even w the first node at or above g.  Worked by hand on
    20 x 12 with bins of 8 x 8 (Sec. III-A), w = 7 and w = 6."""
    n = (20, 12)
    m = (8, 8)
    h1, h2 = 2 * np.pi / 20, 2 * np.pi / 12
    g = [(0.4, 0.6), (7.6, 7.4), (19.7, 11.2), (8.5, 3.0), (15.5, 0.1)]
    x = [a * h1 for a, _ in g]
    y = [b * h2 for _, b in g]
    # w = 7 (odd): index = ceil(g - 3.5) + 3 = ceil(g - 0.5):
    #   (0.4, 0.6) -> (0, 1); (7.6, 7.4) -> (8, 7); (19.7, 11.2) -> (20 = 0, 11);
    #   (8.5, 3.0) -> (8, 3) (the tie 8.5 goes down); (15.5, 0.1) -> (15, 0)
    r = oracle.binsort([x, y], n, m, msub=8, origin_w=7)
    assert list(r["bin_of"]) == [0, 1, 3, 1, 1]
    assert list(r["counts"]) == [1, 3, 0, 1, 0, 0]
    assert list(r["perm"]) == [0, 1, 3, 4, 2]
    # w = 6 (even): index = ceil(g - 3) + 3 = ceil(g):
    #   (0.4, 0.6) -> (1, 1); (7.6, 7.4) -> (8, 8); (19.7, 11.2) -> (20 = 0, 12 = 0);
    #   (8.5, 3.0) -> (9, 3); (15.5, 0.1) -> (16, 1)
    r = oracle.binsort([x, y], n, m, msub=8, origin_w=6)
    assert list(r["bin_of"]) == [0, 4, 0, 1, 2]
    assert list(r["counts"]) == [2, 1, 1, 0, 1, 0]
    assert list(r["perm"]) == [0, 2, 3, 4, 1]
    # cell binning of the same points (origin_w = 0) for contrast
    r = oracle.binsort([x, y], n, m, msub=8)
    assert list(r["bin_of"]) == [0, 0, 5, 1, 1]


def test_binsort_invariants_random():
    rng = np.random.default_rng(3)
    pts = [rng.normal(0, 0.3, 5000) for _ in range(3)]
    n, m = (32, 24, 40), (8, 8, 4)
    r = oracle.binsort(pts, n, m, msub=64)
    assert sorted(r["perm"]) == list(range(5000))
    assert r["counts"].sum() == 5000
    b = r["bin_of"][r["perm"]]
    assert np.all(np.diff(b) >= 0)                     # bin order
    for lo, cnt in zip(r["starts"], r["counts"]):
        seg = r["perm"][lo:lo + cnt]
        assert np.all(np.diff(seg) > 0)                # stable
    t = r["subproblems"]
    assert t[:, 2].max() <= 64 and t[:, 2].sum() == 5000
    assert np.all(t[1:, 1] == t[:-1, 1] + t[:-1, 2])   # contiguous cover


def test_binsort_handpicked_1d():
    """1D: bins of m cells along the only axis; the last bin is smaller."""
    n, m = (20,), (8,)
    h = 2 * np.pi / 20
    x = [c * h for c in (0.5, 19.5, 8.5, 16.2, 7.9)]
    r = oracle.binsort([x], n, m, msub=2)
    assert list(r["bin_of"]) == [0, 2, 1, 2, 0]
    assert list(r["counts"]) == [2, 1, 2]
    assert list(r["perm"]) == [0, 4, 2, 1, 3]


def test_subproblem_split_worked_example():
    """SM step 1: a bin with more than M_sub points is split into chunks of at most M_sub."""
    lib = oracle._load()
    counts = np.array([0, 5, 2048, 1], np.int32)
    starts = np.array([0, 0, 5, 2053], np.int32)
    table = np.zeros((4, 3), np.int32)
    ns = lib.oracle_subproblems(4, oracle._ptr(counts), oracle._ptr(starts), 1024, oracle._ptr(table))
    assert ns == 4
    assert table.tolist() == [[1, 0, 5], [2, 5, 1024], [2, 1029, 1024], [3, 2053, 1]]
