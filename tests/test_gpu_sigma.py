"""Upsampling factor sigma < 2 (nufft_makeplan_upsampled) against the oracle.

"cuFINUFFT: a load-balanced GPU library for general-purpose nonuniform FFTs"
fixes sigma = 2 (Sec. I-B, limitation 3) and names smaller sigma as a way to
save memory and time.  Library and oracle implement the same reading of
eq. (6) for sigma < 2 independently; the plan's width and fine grid must
equal the oracle's, the transforms must match the oracle's three-step NUFFT
at the same sigma and the direct sums within max(2 eps, 1.25 x the oracle
NUFFT's own error, the rounding measure below).

Tolerance against the oracle NUFFT: max(1e-5 / 1e-12, 10 x the oracle's own
change when every coordinate moves by the library's coordinate rounding).
The two sides round coordinates differently: the oracle works with x / h in
double, the library with a coordinate relative to its bin (at most 64 cells
there), rounded to the plan's real type.  So the move is one ulp of pi in
double, 64 * 2^-24 cells in single precision.  At small sigma with a wide
kernel the correction factors p(k) of eq. (10) span up to 1e6, which turns
that rounding into ~1e-11 (double, 2D, sigma = 1.25, w = 16) or a few 1e-5
(single) relative differences; at sigma = 2 the double measure is ~2e-14.
The same amplification applies to the single-precision rounding of the fine
grid itself, so complex64 plans at sigma < 2 are tested at eps >= 1e-4: at
sigma = 1.25 the edge modes of a 3D eps = 1e-5 transform come out near 1e-4."""
import numpy as np
import pytest
import torch

import nonuniform_fft_gb300 as nf
import oracle
from test_gpu_parity import DEV, TOL_O2, _check_direct, _cplx, _dtypes, _pts

pytestmark = pytest.mark.gpu


def _run(ttype, pts, data, N, eps, iflag, dt, sigma, opts):
    cname, rdt, cdt = _dtypes(dt)
    M = len(pts[0])
    xs = [torch.from_numpy(np.ascontiguousarray(p, dtype=rdt)).to(DEV) for p in pts]
    d = torch.from_numpy(np.ascontiguousarray(data, dtype=cdt)).to(DEV)
    out = torch.zeros(int(np.prod(N)) if ttype == 1 else M, dtype=getattr(torch, cname), device=DEV)
    with nf.Plan(ttype, N, iflag, eps, cname, sigma=sigma, **opts) as plan:
        plan.setpts(*xs)
        if ttype == 1:
            plan.execute(d, out)
        else:
            plan.execute(out, d)
        info = plan.info()
        torch.cuda.synchronize()
    return out.cpu().numpy(), info


CASES = [
    # dim, N, dt, eps, sigma, opts
    (1, (1500,), "f32", 1e-4, 1.25, {}),
    (1, (1500,), "f64", 1e-9, 1.5, {}),
    (2, (100, 70), "f32", 1e-4, 1.25, {}),
    (2, (100, 70), "f32", 1e-3, 1.5, {}),
    (2, (100, 70), "f64", 1e-9, 1.25, {}),
    (2, (100, 70), "f64", 1e-12, 1.75, {}),
    (2, (99, 71), "f32", 1e-4, 1.25, {"method": nf.METHOD_SM}),
    (2, (100, 70), "f32", 1e-4, 1.25, {"method": nf.METHOD_GM_SORT}),
    (2, (100, 70), "f64", 1e-6, 1.5, {"method": nf.METHOD_GM}),
    (3, (20, 24, 36), "f32", 1e-4, 1.25, {}),
    (3, (20, 24, 36), "f64", 1e-9, 1.5, {}),
    (3, (21, 24, 35), "f32", 1e-3, 1.25, {"method": nf.METHOD_SM}),
]


@pytest.mark.parametrize("ttype", [1, 2])
@pytest.mark.parametrize("dim,N,dt,eps,sigma,opts", CASES)
def test_sigma_matches_oracle(dim, N, dt, eps, sigma, opts, ttype):
    rng = np.random.default_rng(60 + dim)
    M = 15000
    pts = _pts(dim, M, "uniform", rng, dt)
    iflag = -1 if ttype == 1 else 1
    if ttype == 1:
        data = _cplx(M, rng, dt)
        got, info = _run(1, pts, data, N, eps, iflag, dt, sigma, opts)
        o2 = oracle.nufft_type1(pts, data, N, eps, iflag, sigma).ravel()
        ks = [np.unique(np.concatenate([rng.choice(np.arange(-(n // 2), n - n // 2), min(n, 9),
                                                   replace=False), [0]])) for n in N]
        o1 = oracle.direct_type1(pts, data, N, iflag, modes=ks).ravel()
        sel = np.ix_(*[k + n // 2 for k, n in zip(reversed(ks), reversed(N))])
        sub = lambda a: a.reshape(tuple(reversed(N)))[sel].ravel()  # noqa: E731
    else:
        data = _cplx(int(np.prod(N)), rng, dt)
        got, info = _run(2, pts, data, N, eps, iflag, dt, sigma, opts)
        o2 = oracle.nufft_type2(pts, data, N, eps, iflag, sigma)
        tg = np.arange(0, M, 11)
        o1 = oracle.direct_type2(pts, data, N, iflag, targets=tg)
        sub = lambda a: a[tg]  # noqa: E731
    w, _, n = oracle.plan_params(N, eps, sigma)
    assert info["w"] == w
    assert [info["n1"], info["n2"], info["n3"]][:dim] == list(n)
    assert any(ni < 2 * Ni for ni, Ni in zip(n, N))      # a smaller grid than sigma = 2
    step = [np.spacing(np.pi) if dt == "f64" else 64 * 2.0 ** -24 * 2 * np.pi / ni for ni in n]
    moved = [np.asarray(x, np.float64) + rng.choice([-1.0, 1.0], M) * s_d
             for x, s_d in zip(pts, step)]
    o2m = (oracle.nufft_type1(moved, data, N, eps, iflag, sigma).ravel() if ttype == 1
           else oracle.nufft_type2(moved, data, N, eps, iflag, sigma))
    assert oracle.rel_l2(got, o2) <= max(TOL_O2[dt], 10 * oracle.rel_l2(o2m, o2))
    # the same rounding bounds the reachable accuracy on the sampled outputs
    sens = 10 * oracle.rel_l2(sub(o2m), sub(o2))
    err, err_o2 = oracle.rel_l2(sub(got), o1), oracle.rel_l2(sub(o2), o1)
    if err > sens:
        _check_direct(err, err_o2, eps)


def test_sigma_two_is_makeplan():
    """sigma = 2 through the upsampled entry point equals nufft_makeplan."""
    import ctypes
    lib = nf.load_library()
    arr = (ctypes.c_int64 * 2)(100, 70)
    h = ctypes.c_void_p()
    assert lib.nufft_makeplan_upsampled(1, 2, arr, -1, 1e-6, 0, 2.0, None, ctypes.byref(h)) == nf.OK
    a = nf.get_info(h.value)
    nf.destroy(h.value)
    with nf.Plan(1, (100, 70), -1, 1e-6) as plan:
        b = plan.info()
    assert a == b and a["w"] == 7 and (a["n1"], a["n2"]) == (200, 144)
