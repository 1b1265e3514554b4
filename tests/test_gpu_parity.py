"""CUDA path against the CPU oracle, element by element, through the C ABI.

Tolerances (the method's own, see "cuFINUFFT: a load-balanced GPU library for
general-purpose nonuniform FFTs", Sec. II):
  * GPU vs the oracle's three-step NUFFT with identical parameters, relative
    l2: 1e-5 for complex64, 1e-12 for complex128 (only rounding differs);
  * GPU vs the direct sums of eq. (1) / eq. (3): at most 2 eps, and never
    more than 25 % above the oracle NUFFT's own error on the same outputs
    (the method's error is "close to eps": about 3 eps for w = 13 in 3D);
  * integer setpts results (bin counts, starts, subproblem table): identical
    to the oracle's counting sort; the order of points inside a bin is not
    unique, so the permutation is compared bin by bin as a set.
"""
import numpy as np
import pytest
import torch

import nonuniform_fft_gb300 as nf
import oracle
from nonuniform_fft_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
TOL_O2 = {"f32": 1e-5, "f64": 1e-12}


def _dtypes(dt):
    return ("complex64", np.float32, np.complex64) if dt == "f32" else \
        ("complex128", np.float64, np.complex128)


def gpu_transform(ttype, pts, data, N, eps, iflag, dt, opts=None, host=False, plan_out=None):
    """Run one transform through the C ABI; returns a numpy array (f shaped
    (N3,) N2, N1 for type 1; c of length M for type 2)."""
    cname, rdt, cdt = _dtypes(dt)
    M = len(pts[0])
    if host:
        xs = [np.ascontiguousarray(p, dtype=rdt) for p in pts]
        d = np.ascontiguousarray(data, dtype=cdt)
        out = np.zeros(tuple(reversed(N)) if ttype == 1 else (M,), dtype=cdt)
    else:
        xs = [torch.from_numpy(np.ascontiguousarray(p, dtype=rdt)).to(DEV) for p in pts]
        d = torch.from_numpy(np.ascontiguousarray(data, dtype=cdt)).to(DEV)
        out = torch.zeros(tuple(reversed(N)) if ttype == 1 else (M,), dtype=getattr(torch, cname),
                          device=DEV)
    with nf.Plan(ttype, N, iflag, eps, cname, **(opts or {})) as plan:
        plan.setpts(*xs)
        if ttype == 1:
            plan.execute(d, out)
        else:
            plan.execute(out, d)
        if plan_out is not None:
            plan_out.update(plan.info())
            plan_out["timings"] = plan.timings()
        torch.cuda.synchronize()
    return out if host else out.cpu().numpy()


def _pts(dim, M, dist, rng, dt):
    _, rdt, _ = _dtypes(dt)
    if dist == "uniform":
        return [rng.uniform(-np.pi, np.pi, M).astype(rdt) for _ in range(dim)]
    if dist == "cluster":
        return [(np.mod(rng.normal(0, 0.05, M) + np.pi, 2 * np.pi) - np.pi).astype(rdt)
                for _ in range(dim)]
    if dist == "wild":   # far outside [-pi, pi) and on the fold boundaries
        v = [rng.uniform(-40, 40, M) for _ in range(dim)]
        for a in v:
            a[: min(6, M)] = [-np.pi, np.pi, 2 * np.pi, -1e-300, 0.0, 3 * np.pi][: min(6, M)]
        return [a.astype(rdt) for a in v]
    raise ValueError(dist)


def _cplx(n, rng, dt):
    _, _, cdt = _dtypes(dt)
    return (rng.standard_normal(n) + 1j * rng.standard_normal(n)).astype(cdt)


def _check_direct(err_gpu, err_o2, eps):
    bound = max(2 * eps, 1.25 * err_o2)
    assert err_gpu <= bound, f"GPU vs direct {err_gpu:.3e} > {bound:.3e} (oracle NUFFT {err_o2:.3e})"


# ---------------------------------------------------------------- setpts

SORT_CASES = [
    # dim, N, M, dist, dt, opts
    (1, (3000,), 20000, "cluster", "f32", {}),
    (1, (3000,), 20000, "uniform", "f64", {"msub": 64}),
    (2, (100, 70), 20000, "uniform", "f32", {"msub": 256}),
    (2, (100, 70), 20000, "cluster", "f32", {"msub": 100}),
    (2, (64, 64), 5000, "wild", "f64", {}),
    (2, (64, 64), 5000, "wild", "f32", {}),
    (3, (20, 24, 36), 30000, "uniform", "f32", {"bin1": 8, "bin2": 8, "bin3": 4, "msub": 128}),
    (3, (20, 24, 36), 30000, "cluster", "f64", {}),
    (2, (3, 5), 50, "uniform", "f32", {"bin1": 5, "bin2": 7}),
]


@pytest.mark.parametrize("dim,N,M,dist,dt,opts", SORT_CASES)
def test_setpts_integer_results_match_oracle(dim, N, M, dist, dt, opts):
    rng = np.random.default_rng(11)
    pts = _pts(dim, M, dist, rng, dt)
    cname, rdt, _ = _dtypes(dt)
    xs = [torch.from_numpy(p).to(DEV) for p in pts]
    with nf.Plan(1, N, -1, 1e-6 if dt == "f32" else 1e-12, cname, **opts) as plan:
        plan.setpts(*xs)
        info = plan.info()
        got = plan.sort()
    n = [info["n1"], info["n2"], info["n3"]][:dim]
    m = [info["bin1"], info["bin2"], info["bin3"]][:dim]
    # the 3D single-precision slab spreader bins by window origin
    origin_w = info["w"] if info["bin_origin"] else 0
    assert info["bin_origin"] == (dim == 3 and info["tile3d"] == 2)
    ref = oracle.binsort(pts, n, m, info["msub"], origin_w=origin_w)
    assert info["nbins"] == ref["counts"].size
    np.testing.assert_array_equal(got["counts"], ref["counts"])
    np.testing.assert_array_equal(got["starts"], ref["starts"])
    np.testing.assert_array_equal(got["subproblems"], ref["subproblems"])
    for lo, cnt in zip(ref["starts"], ref["counts"]):
        np.testing.assert_array_equal(np.sort(got["perm"][lo:lo + cnt]), ref["perm"][lo:lo + cnt])


def _boundary_coords(n, rng, count, offset=0.0):
    """float32 coordinates at and next to the floats nearest the cell
    boundaries 2 pi (k + offset) / n, one period either side too, in random
    order."""
    k = rng.integers(0, n + 1, count).astype(np.float64) + offset
    shift = rng.choice([0.0, -2 * np.pi, 2 * np.pi], count)
    b = (2 * np.pi * k / n + shift).astype(np.float32)
    step = rng.integers(-2, 3, count)
    for s in (1, 2):
        b = np.where(step >= s, np.nextafter(b, np.float32(np.inf)), b)
        b = np.where(step <= -s, np.nextafter(b, np.float32(-np.inf)), b)
    return b


@pytest.mark.parametrize("eps", [1e-6, 1e-5, 1e-7])
def test_setpts_origins_at_boundaries_match_oracle(eps):
    """The slab spreader's plans bin points by window origin (ceil(g - w/2)
    + floor(w/2)): with bins one origin high in y and z, the bin of a point
    is its y and z origin.  Coordinates at (or next to) the floats nearest
    the origin boundaries -- half-integer g for odd w (w = 7), integer g for
    even w (w = 6, 8) -- must get the oracle's double-precision origins."""
    rng = np.random.default_rng(6)
    M = 60000
    N = (20, 24, 18)
    with nf.Plan(1, N, -1, eps, "complex64", bin2=1) as plan:
        info0 = plan.info()
        w = info0["w"]
        n = [info0["n1"], info0["n2"], info0["n3"]]
        off = 0.5 if w % 2 else 0.0
        pts = [rng.uniform(-np.pi, np.pi, M).astype(np.float32),
               _boundary_coords(n[1], rng, M, off), _boundary_coords(n[2], rng, M, off)]
        plan.setpts(*[torch.from_numpy(p).to(DEV) for p in pts])
        info = plan.info()
        got = plan.sort()
    assert info["tile3d"] == 2 and info["bin_origin"] == 1 and info["bin2"] == 1 and info["bin3"] == 1
    m = [info["bin1"], info["bin2"], info["bin3"]]
    ref = oracle.binsort(pts, n, m, info["msub"], origin_w=w)
    np.testing.assert_array_equal(got["counts"], ref["counts"])
    np.testing.assert_array_equal(got["subproblems"], ref["subproblems"])
    for lo, cnt in zip(ref["starts"], ref["counts"]):
        np.testing.assert_array_equal(np.sort(got["perm"][lo:lo + cnt]), ref["perm"][lo:lo + cnt])


@pytest.mark.parametrize("N", [(100, 70), (64, 128)])
def test_setpts_cells_at_boundaries_match_oracle(N):
    """Single-cell bins make each point's bin its fine-grid cell: with every
    coordinate at (or next to) the float nearest a cell boundary, the cells
    setpts assigns must be the oracle's double-precision fold's."""
    rng = np.random.default_rng(5)
    M = 60000
    with nf.Plan(1, N, -1, 1e-6, "complex64", method=nf.METHOD_SM, bin1=1, bin2=1) as plan:
        n = [plan.info()["n1"], plan.info()["n2"]]
        pts = [_boundary_coords(nd, rng, M) for nd in n]
        plan.setpts(*[torch.from_numpy(p).to(DEV) for p in pts])
        info = plan.info()
        got = plan.sort()
    assert info["bin1"] == 1 and info["bin2"] == 1
    ref = oracle.binsort(pts, n, [1, 1], info["msub"])
    np.testing.assert_array_equal(got["counts"], ref["counts"])
    for lo, cnt in zip(ref["starts"], ref["counts"]):
        np.testing.assert_array_equal(np.sort(got["perm"][lo:lo + cnt]), ref["perm"][lo:lo + cnt])


# ---------------------------------------------------------------- transforms

T_CASES = []
for _dim, _N in ((1, (1500,)), (2, (100, 70)), (3, (20, 24, 36))):
    for _dt, _epss in (("f32", (1e-2, 1e-5, 1e-6)), ("f64", (1e-3, 1e-9, 1e-12))):
        for _eps in _epss:
            T_CASES.append((_dim, _N, _dt, _eps))


METHODS = [nf.METHOD_SM, nf.METHOD_GM_SORT, nf.METHOD_REGTILE, nf.METHOD_GM]


@pytest.mark.parametrize("cols", [1, 2, 4])
@pytest.mark.parametrize("dt,eps", [("f32", 1e-2), ("f32", 1e-6), ("f64", 1e-9), ("f64", 1e-12)])
@pytest.mark.parametrize("rows", [0, 13, 128])
def test_regtile_columns_per_lane(cols, dt, eps, rows):
    """The register-tile spreader with 1, 2 and 4 tile columns per lane and
    bin heights of 13, 64 (default) and 128 rows, on a grid whose sizes are
    not multiples of the bin (ragged last bins)."""
    rng = np.random.default_rng(31)
    N = (150, 90)
    M = 30000
    pts = _pts(2, M, "uniform", rng, dt)
    c = _cplx(M, rng, dt)
    opts = {"method": nf.METHOD_REGTILE, "regtile_cols": cols, "msub": 700}
    if rows:
        opts["bin2"] = rows
    f = gpu_transform(1, pts, c, N, eps, -1, dt, opts)
    assert oracle.rel_l2(f, oracle.nufft_type1(pts, c, N, eps, -1)) <= TOL_O2[dt]


@pytest.mark.parametrize("eps", [1e-2, 1e-5, 1e-6, 1e-7])
@pytest.mark.parametrize("N,dist,opts", [((20, 24, 36), "uniform", {}),
                                         ((33, 18, 16), "cluster", {}),
                                         ((20, 24, 36), "uniform", {"msub": 37, "bin2": 5}),
                                         ((20, 24, 36), "wild", {})])
def test_slab3d_spreader(eps, N, dist, opts):
    """The 3D single-precision spreader with one-cell-thick bins (option
    tile3d = 2; widths 3, 6, 7 and 8 here), ragged grids, clustered points
    and short subproblems, against the oracle's three-step NUFFT."""
    rng = np.random.default_rng(41)
    M = 40000
    pts = _pts(3, M, dist, rng, "f32")
    c = _cplx(M, rng, "f32")
    info = {}
    f = gpu_transform(1, pts, c, N, eps, -1, "f32",
                      dict(opts, method=nf.METHOD_REGTILE, tile3d=2), plan_out=info)
    assert info["bin3"] == 1
    assert oracle.rel_l2(f, oracle.nufft_type1(pts, c, N, eps, -1)) <= TOL_O2["f32"]


@pytest.mark.parametrize("eps", [1e-3, 1e-6])
@pytest.mark.parametrize("dist", ["uniform", "cluster"])
def test_plane3d_spreader_single_precision(eps, dist):
    """The 3D single-precision spreader with planes per warp (option tile3d =
    1; the default where slab bins do not apply, w > 8)."""
    rng = np.random.default_rng(43)
    N = (20, 24, 36)
    M = 40000
    pts = _pts(3, M, dist, rng, "f32")
    c = _cplx(M, rng, "f32")
    info = {}
    f = gpu_transform(1, pts, c, N, eps, -1, "f32", {"method": nf.METHOD_REGTILE, "tile3d": 1},
                      plan_out=info)
    assert info["tile3d"] == 1 and info["bin3"] > 1
    assert oracle.rel_l2(f, oracle.nufft_type1(pts, c, N, eps, -1)) <= TOL_O2["f32"]


def test_slab3d_rejects_unsupported():
    """Slab bins are built for single precision and widths up to 8."""
    x = torch.zeros(10, dtype=torch.float64, device=DEV)
    with nf.Plan(1, (8, 8, 8), -1, 1e-9, "complex128", method=nf.METHOD_REGTILE, tile3d=2) as plan:
        with pytest.raises(nf.NufftError) as e:
            plan.setpts(x, x, x)
        assert e.value.code == nf.ERR_BAD_OPT
    xf = torch.zeros(10, dtype=torch.float32, device=DEV)
    with nf.Plan(1, (8, 8, 8), -1, 1e-9, "complex64", method=nf.METHOD_REGTILE, tile3d=2) as plan:
        with pytest.raises(nf.NufftError) as e:      # w = 10
            plan.setpts(xf, xf, xf)
        assert e.value.code == nf.ERR_BAD_OPT


@pytest.mark.parametrize("method", METHODS)
@pytest.mark.parametrize("dim,N,dt,eps", T_CASES)
def test_type1_matches_oracle(dim, N, dt, eps, method):
    if dim == 1 and method in (nf.METHOD_GM, nf.METHOD_GM_SORT):
        pytest.skip("1D has the register-tile spreader and the shared-memory interpolator")
    rng = np.random.default_rng(21)
    M = 20000
    pts = _pts(dim, M, "uniform", rng, dt)
    c = _cplx(M, rng, dt)
    for iflag in (-1, 1):
        f = gpu_transform(1, pts, c, N, eps, iflag, dt, {"method": method, "msub": 300})
        o2 = oracle.nufft_type1(pts, c, N, eps, iflag)
        o1 = oracle.direct_type1(pts, c, N, iflag)
        e = oracle.rel_l2(f, o2)
        assert e <= TOL_O2[dt], f"GPU vs oracle NUFFT {e:.3e}"
        _check_direct(oracle.rel_l2(f, o1), oracle.rel_l2(o2, o1), eps)


@pytest.mark.parametrize("method", METHODS)
@pytest.mark.parametrize("dim,N,dt,eps", T_CASES)
def test_type2_matches_oracle(dim, N, dt, eps, method):
    if dim == 1 and method in (nf.METHOD_GM, nf.METHOD_GM_SORT):
        pytest.skip("1D has the register-tile spreader and the shared-memory interpolator")
    rng = np.random.default_rng(22)
    M = 20000
    pts = _pts(dim, M, "uniform", rng, dt)
    f = _cplx(int(np.prod(N)), rng, dt)
    for iflag in (-1, 1):
        c = gpu_transform(2, pts, f, N, eps, iflag, dt, {"method": method, "msub": 300})
        o2 = oracle.nufft_type2(pts, f, N, eps, iflag)
        tg = np.arange(0, M, 7)
        o1 = oracle.direct_type2(pts, f, N, iflag, targets=tg)
        e = oracle.rel_l2(c, o2)
        assert e <= TOL_O2[dt], f"GPU vs oracle NUFFT {e:.3e}"
        _check_direct(oracle.rel_l2(c[tg], o1), oracle.rel_l2(o2[tg], o1), eps)


@pytest.mark.parametrize("dim,N,dt", [(2, (48, 40), "f32"), (3, (12, 10, 16), "f64")])
def test_adjoint_identity_on_gpu(dim, N, dt):
    """<T1_s(c), f> = <c, T2_-s(f)> holds to rounding for the GPU transforms."""
    rng = np.random.default_rng(5)
    M = 5000
    pts = _pts(dim, M, "uniform", rng, dt)
    c = _cplx(M, rng, dt).astype(np.complex128)
    f = _cplx(int(np.prod(N)), rng, dt).astype(np.complex128)
    for s in (-1, 1):
        t1 = gpu_transform(1, pts, c, N, 1e-6 if dt == "f32" else 1e-12, s, dt).astype(np.complex128)
        t2 = gpu_transform(2, pts, f, N, 1e-6 if dt == "f32" else 1e-12, -s, dt).astype(np.complex128)
        lhs = np.vdot(t1.ravel(), f)
        rhs = np.vdot(c, t2)
        tol = 1e-5 if dt == "f32" else 1e-12
        assert abs(lhs - rhs) <= tol * abs(lhs)


@pytest.mark.parametrize("method", METHODS)
def test_clustered_points_single_bin(method):
    """Every point in one fine cell: one bin, many subproblems (SM step 1
    load balancing), heavy atomic contention."""
    rng = np.random.default_rng(9)
    M = 50000
    h = 2 * np.pi / 256
    pts = [(0.3 + rng.uniform(0, h, M)).astype(np.float32) for _ in range(2)]
    c = _cplx(M, rng, "f32")
    info = {}
    f = gpu_transform(1, pts, c, (128, 128), 1e-5, -1, "f32", {"method": method}, plan_out=info)
    if method != nf.METHOD_GM:  # GM has no subproblems
        assert info["nsub"] >= M // 2048
    ref = oracle.nufft_type1(pts, c, (128, 128), 1e-5, -1)
    assert oracle.rel_l2(f, ref) <= 1e-5


@pytest.mark.parametrize("dt,eps", [("f32", 1e-6), ("f64", 1e-12), ("f64", 1e-3)])
@pytest.mark.parametrize("msub", [100000, 500])
def test_regtile3d_clustered_and_ragged(dt, eps, msub):
    """3D register-tile spreading on a grid that is not a multiple of the bin
    (ragged last bins in every dimension), with a cluster that puts many
    subproblems in a few bins."""
    rng = np.random.default_rng(41)
    N = (30, 22, 26)
    M = 40000
    pts = _pts(3, M, "uniform", rng, dt)
    for a in pts:
        a[: M // 2] = (np.mod(rng.normal(0.5, 0.08, M // 2) + np.pi, 2 * np.pi) - np.pi).astype(a.dtype)
    c = _cplx(M, rng, dt)
    f = gpu_transform(1, pts, c, N, eps, 1, dt, {"method": nf.METHOD_REGTILE, "msub": msub})
    assert oracle.rel_l2(f, oracle.nufft_type1(pts, c, N, eps, 1)) <= TOL_O2[dt]


@pytest.mark.parametrize("N", [(1,), (3,), (1, 1), (2, 3), (1, 4, 2)])
def test_tiny_mode_counts(N):
    """Fine grid of 2w points per dimension: the padded tile wraps onto itself."""
    rng = np.random.default_rng(4)
    pts = _pts(len(N), 300, "uniform", rng, "f64")
    c = _cplx(300, rng, "f64")
    f = gpu_transform(1, pts, c, N, 1e-9, 1, "f64")
    assert oracle.rel_l2(f, oracle.nufft_type1(pts, c, N, 1e-9, 1)) <= 1e-12
    fk = _cplx(int(np.prod(N)), rng, "f64")
    c2 = gpu_transform(2, pts, fk, N, 1e-9, -1, "f64")
    assert oracle.rel_l2(c2, oracle.nufft_type2(pts, fk, N, 1e-9, -1)) <= 1e-12


def test_wild_coordinates_fold():
    rng = np.random.default_rng(6)
    pts = _pts(2, 4000, "wild", rng, "f64")
    c = _cplx(4000, rng, "f64")
    f = gpu_transform(1, pts, c, (30, 22), 1e-12, -1, "f64")
    assert oracle.rel_l2(f, oracle.nufft_type1(pts, c, (30, 22), 1e-12, -1)) <= 1e-12


def test_host_pointers_match_device_pointers():
    rng = np.random.default_rng(8)
    pts = _pts(2, 3000, "uniform", rng, "f32")
    c = _cplx(3000, rng, "f32")
    fd = gpu_transform(1, pts, c, (40, 24), 1e-5, -1, "f32")
    fh = gpu_transform(1, pts, c, (40, 24), 1e-5, -1, "f32", host=True)
    assert oracle.rel_l2(fh, fd) <= 1e-6
    fk = _cplx(40 * 24, rng, "f32")
    cd = gpu_transform(2, pts, fk, (40, 24), 1e-5, 1, "f32")
    ch = gpu_transform(2, pts, fk, (40, 24), 1e-5, 1, "f32", host=True)
    assert oracle.rel_l2(ch, cd) <= 1e-6


def test_zero_points():
    f = gpu_transform(1, [np.zeros(0), np.zeros(0)], np.zeros(0), (16, 8), 1e-6, -1, "f32")
    assert f.shape == (8, 16) and np.all(f == 0)
    c = gpu_transform(2, [np.zeros(0), np.zeros(0)], np.ones(128), (16, 8), 1e-6, 1, "f32")
    assert c.shape == (0,)


def test_single_point_closed_form():
    N = (33, 20)
    x0 = [np.array([-np.pi]), np.array([1.234])]
    f = gpu_transform(1, x0, np.ones(1), N, 1e-12, -1, "f64")
    k1 = np.arange(-(N[0] // 2), N[0] - N[0] // 2)[None, :]
    k2 = np.arange(-(N[1] // 2), N[1] - N[1] // 2)[:, None]
    ref = np.exp(-1j * (k1 * x0[0][0] + k2 * x0[1][0]))
    assert oracle.rel_l2(f, ref) <= 20e-12


def test_errors_reported():
    xs = [torch.tensor([0.1, float("nan")], device=DEV), torch.tensor([0.0, 0.2], device=DEV)]
    plan = nf.Plan(1, (8, 8), -1, 1e-5, "complex64")
    try:
        with pytest.raises(nf.NufftError) as ei:
            plan.execute(torch.zeros(2, dtype=torch.complex64, device=DEV),
                         torch.zeros(64, dtype=torch.complex64, device=DEV))
        assert ei.value.code == nf.ERR_NO_POINTS
        with pytest.raises(nf.NufftError) as ei:
            plan.setpts(*xs)
        assert ei.value.code == nf.ERR_BAD_POINTS
        with pytest.raises(nf.NufftError) as ei:
            plan.set_opt("no_such_key", 1)
        assert ei.value.code == nf.ERR_BAD_OPT
        with pytest.raises(nf.NufftError) as ei:
            plan.set_opt("threads", 33)
        assert ei.value.code == nf.ERR_BAD_OPT
        # too-large bins for shared memory are refused at setpts
        big = [torch.zeros(4, device=DEV), torch.zeros(4, device=DEV)]
        p2 = nf.Plan(1, (2048, 2048), -1, 1e-5, "complex64", bin1=1024, bin2=1024,
                     method=nf.METHOD_SM)
        with pytest.raises(nf.NufftError) as ei:
            p2.setpts(*big)
        assert ei.value.code == nf.ERR_BAD_OPT
        p2.close()

    finally:
        plan.close()


def test_1d_rejects_other_methods():
    xs = [torch.zeros(8, device=DEV)]
    with nf.Plan(1, (8,), -1, 1e-5, "complex64", method=nf.METHOD_GM) as plan:
        with pytest.raises(nf.NufftError) as ei:
            plan.setpts(*xs)
        assert ei.value.code == nf.ERR_BAD_OPT


def test_gm_has_no_sort():
    xs = [torch.zeros(8, device=DEV), torch.zeros(8, device=DEV)]
    with nf.Plan(1, (8, 8), -1, 1e-5, "complex64", method=nf.METHOD_GM) as plan:
        plan.setpts(*xs)
        with pytest.raises(nf.NufftError) as ei:
            plan.sort()
        assert ei.value.code == nf.ERR_BAD_OPT


def test_plan_reuse_new_strengths_and_points():
    """One plan, several setpts and executes (Sec. I-A 'plan, setup, execute')."""
    rng = np.random.default_rng(12)
    N = (50, 36)
    with nf.Plan(1, N, -1, 1e-6, "complex64") as plan:
        for M in (5000, 20000, 700):
            pts = _pts(2, M, "uniform", rng, "f32")
            plan.setpts(*[torch.from_numpy(p).to(DEV) for p in pts])
            for _ in range(2):
                c = _cplx(M, rng, "f32")
                f = torch.zeros(N[1], N[0], dtype=torch.complex64, device=DEV)
                plan.execute(torch.from_numpy(c).to(DEV), f)
                ref = oracle.nufft_type1(pts, c, N, 1e-6, -1)
                assert oracle.rel_l2(f.cpu().numpy(), ref) <= 1e-5


@pytest.mark.parametrize("dim,N", [(1, (700,)), (2, (60, 44)), (3, (16, 12, 20))])
@pytest.mark.parametrize("eps", [1e-14, 1e-15])
@pytest.mark.parametrize("ttype", [1, 2])
def test_widest_kernels(dim, N, eps, ttype):
    """w = 15 and 16 (eq. (6) at eps = 1e-14, 1e-15), the widest the library
    accepts, in double precision: against the oracle NUFFT at 1e-12 and the
    direct sums at the double-precision floor (1e-12)."""
    rng = np.random.default_rng(23)
    M = 6000
    pts = _pts(dim, M, "uniform", rng, "f64")
    iflag = 1 if ttype == 1 else -1
    if ttype == 1:
        c = _cplx(M, rng, "f64")
        f = gpu_transform(1, pts, c, N, eps, iflag, "f64")
        assert oracle.rel_l2(f, oracle.nufft_type1(pts, c, N, eps, iflag)) <= 1e-12
        assert oracle.rel_l2(f, oracle.direct_type1(pts, c, N, iflag)) <= 1e-12
    else:
        fk = _cplx(int(np.prod(N)), rng, "f64")
        c = gpu_transform(2, pts, fk, N, eps, iflag, "f64")
        assert oracle.rel_l2(c, oracle.nufft_type2(pts, fk, N, eps, iflag)) <= 1e-12
        tg = np.arange(0, M, 13)
        assert oracle.rel_l2(c[tg], oracle.direct_type2(pts, fk, N, iflag, targets=tg)) <= 1e-12


def test_threads_option_is_lowered_to_what_a_kernel_allows():
    """1024 threads per block exceed the register budget of some kernels; the
    launch uses the most the kernel allows instead of failing."""
    rng = np.random.default_rng(24)
    N = (12, 10, 8)
    pts = _pts(3, 3000, "uniform", rng, "f64")
    fk = _cplx(int(np.prod(N)), rng, "f64")
    for method in (nf.METHOD_SM, nf.METHOD_GM_SORT):
        c = gpu_transform(2, pts, fk, N, 1e-9, 1, "f64", {"threads": 1024, "method": method})
        assert oracle.rel_l2(c, oracle.nufft_type2(pts, fk, N, 1e-9, 1)) <= 1e-12


@pytest.mark.parametrize("dim,N", [(1, (700,)), (2, (70, 46)), (3, (30, 22, 26))])
@pytest.mark.parametrize("dt,eps", [("f32", 1e-5), ("f64", 1e-12)])
@pytest.mark.parametrize("msub", [0, 37])
def test_interp_clustered_and_ragged(dim, N, dt, eps, msub):
    """Type 2 with half the points in one cluster (many subproblems in a few
    bins), grids that are not a multiple of the bin size, and an odd M_sub
    (subproblems of 37 points: the 3D single-precision interpolator walks its
    bank-sorted points with a stride coprime with 37)."""
    rng = np.random.default_rng(43)
    M = 30000
    pts = _pts(dim, M, "uniform", rng, dt)
    for a in pts:
        a[: M // 2] = (np.mod(rng.normal(-1.0, 0.05, M // 2) + np.pi, 2 * np.pi) - np.pi).astype(a.dtype)
    fk = _cplx(int(np.prod(N)), rng, dt)
    opts = {"msub": msub} if msub else {}
    c = gpu_transform(2, pts, fk, N, eps, 1, dt, opts)
    assert oracle.rel_l2(c, oracle.nufft_type2(pts, fk, N, eps, 1)) <= TOL_O2[dt]


def test_interp3d_large_msub_is_capped():
    """A 3D type 2 plan asked for huge subproblems interpolates with at most
    8192 points per subproblem (its per-block point order lives next to the
    tile in shared memory) and still matches the oracle."""
    rng = np.random.default_rng(44)
    N = (16, 20, 12)
    M = 30000
    pts = _pts(3, M, "cluster", rng, "f32")
    fk = _cplx(int(np.prod(N)), rng, "f32")
    info = {}
    c = gpu_transform(2, pts, fk, N, 1e-5, 1, "f32", {"msub": 100000}, plan_out=info)
    assert info["msub"] == 8192
    assert oracle.rel_l2(c, oracle.nufft_type2(pts, fk, N, 1e-5, 1)) <= TOL_O2["f32"]


def _stacked_pts(M, rng, nodes=5):
    """3D points piled on a few spots (each spot's points share one window
    origin, so one origin holds far more than a group's K points), plus a
    uniform half."""
    spots = rng.uniform(-np.pi, np.pi, (3, nodes))
    pick = rng.integers(0, nodes, M // 2)
    pts = []
    for d in range(3):
        a = rng.uniform(-np.pi, np.pi, M)
        a[: M // 2] = spots[d][pick] + rng.uniform(-1e-4, 1e-4, M // 2)
        pts.append(a.astype(np.float32))
    return pts


@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("eps", [1e-2, 1e-5, 1e-6, 1e-7])
@pytest.mark.parametrize("N,dist,opts", [((20, 24, 36), "uniform", {}),
                                         ((33, 18, 16), "cluster", {}),
                                         ((30, 22, 26), "stacked", {"msub": 37}),
                                         ((20, 24, 36), "uniform", {"msub": 8192, "bin1": 7, "bin2": 9,
                                                                   "bin3": 5})])
def test_group3d_interp(K, eps, N, dist, opts):
    """3D single-precision interpolation with the points of one window origin
    in groups of at most K per thread (option igroup; widths 3, 6, 7 and 8
    here): against the oracle's three-step NUFFT, and bit for bit against
    one thread per point (igroup = 1), which sums the same products in the
    same order."""
    rng = np.random.default_rng(47)
    M = 40000
    pts = _stacked_pts(M, rng) if dist == "stacked" else _pts(3, M, dist, rng, "f32")
    fk = _cplx(int(np.prod(N)), rng, "f32")
    info = {}
    c = gpu_transform(2, pts, fk, N, eps, 1, "f32", dict(opts, igroup=K), plan_out=info)
    assert info["igroup"] == K
    assert oracle.rel_l2(c, oracle.nufft_type2(pts, fk, N, eps, 1)) <= TOL_O2["f32"]
    info1 = {}
    c1 = gpu_transform(2, pts, fk, N, eps, 1, "f32", dict(opts, igroup=1), plan_out=info1)
    assert info1["igroup"] == 1
    np.testing.assert_array_equal(c, c1)


@pytest.mark.parametrize("M", [1, 3, 33])
def test_group3d_interp_few_points(M):
    """Subproblems of one to a few dozen points (most groups of one point,
    most warps partly empty)."""
    rng = np.random.default_rng(48)
    N = (16, 12, 10)
    pts = _pts(3, M, "uniform", rng, "f32")
    fk = _cplx(int(np.prod(N)), rng, "f32")
    c = gpu_transform(2, pts, fk, N, 1e-6, -1, "f32", {"igroup": 4})
    assert oracle.rel_l2(c, oracle.nufft_type2(pts, fk, N, 1e-6, -1)) <= TOL_O2["f32"]


def test_group3d_interp_defaults_and_rejection():
    """Grouped interpolation is the default for 3D single-precision type 2
    plans with w <= 8 (groups of 2); other plans report igroup 0; asking for
    groups where the kernel cannot run (w = 10) fails at setpts."""
    xf = torch.zeros(10, dtype=torch.float32, device=DEV)
    with nf.Plan(2, (8, 8, 8), 1, 1e-6, "complex64") as plan:
        plan.setpts(xf, xf, xf)
        assert plan.info()["igroup"] == 2
    with nf.Plan(2, (8, 8, 8), 1, 1e-9, "complex64") as plan:     # w = 10
        plan.setpts(xf, xf, xf)
        assert plan.info()["igroup"] == 1
    with nf.Plan(1, (8, 8, 8), 1, 1e-6, "complex64") as plan:
        plan.setpts(xf, xf, xf)
        assert plan.info()["igroup"] == 0
    with nf.Plan(2, (8, 8, 8), 1, 1e-9, "complex64", igroup=3) as plan:
        with pytest.raises(nf.NufftError) as e:
            plan.setpts(xf, xf, xf)
        assert e.value.code == nf.ERR_BAD_OPT


def test_group3d_interp_plan_reuse():
    """One grouped 3D plan, setpts with more, fewer and again more points
    (the group records are rebuilt, and their storage grown, each time)."""
    rng = np.random.default_rng(49)
    N = (18, 20, 16)
    with nf.Plan(2, N, 1, 1e-6, "complex64") as plan:
        for M in (20000, 700, 45000):
            pts = _pts(3, M, "uniform", rng, "f32")
            plan.setpts(*[torch.from_numpy(p).to(DEV) for p in pts])
            assert plan.info()["igroup"] == 2
            for _ in range(2):
                fk = _cplx(int(np.prod(N)), rng, "f32")
                c = torch.zeros(M, dtype=torch.complex64, device=DEV)
                plan.execute(c, torch.from_numpy(fk).to(DEV))
                ref = oracle.nufft_type2(pts, fk, N, 1e-6, 1)
                assert oracle.rel_l2(c.cpu().numpy(), ref) <= TOL_O2["f32"]
