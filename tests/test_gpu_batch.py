"""Batched execute (nufft_execute_batch): several strength vectors on the
points of one setpts, the reuse that motivates the plan / setup / execute
interface of "cuFINUFFT: a load-balanced GPU library for general-purpose
nonuniform FFTs" (Sec. I).  Every vector is an independent transform, so each
is checked against the oracle's three-step NUFFT of that vector alone
(1e-5 / 1e-12 relative l2) and against the single-vector execute (rounding of
the atomic summation order only)."""
import numpy as np
import pytest
import torch

import nonuniform_fft_gb300 as nf
import oracle
from test_gpu_parity import DEV, TOL_O2, _cplx, _dtypes, _pts

pytestmark = pytest.mark.gpu

SAME = {"f32": 2e-6, "f64": 1e-14}   # batched vs one-by-one, relative l2


def _run_batch(ttype, pts, data, N, eps, iflag, dt, nvec, opts, host=False):
    """data: (nvec, M) strengths (type 1) or (nvec, modes) coefficients."""
    cname, rdt, cdt = _dtypes(dt)
    M = len(pts[0])
    modes = int(np.prod(N))
    out_len = modes if ttype == 1 else M
    if host:
        xs = [np.ascontiguousarray(p, dtype=rdt) for p in pts]
        d = np.ascontiguousarray(data, dtype=cdt)
        out = np.zeros((nvec, out_len), dtype=cdt)
    else:
        xs = [torch.from_numpy(np.ascontiguousarray(p, dtype=rdt)).to(DEV) for p in pts]
        d = torch.from_numpy(np.ascontiguousarray(data, dtype=cdt)).to(DEV)
        out = torch.zeros((nvec, out_len), dtype=getattr(torch, cname), device=DEV)
    with nf.Plan(ttype, N, iflag, eps, cname, **opts) as plan:
        plan.setpts(*xs)
        if ttype == 1:
            plan.execute_batch(nvec, d, out)
        else:
            plan.execute_batch(nvec, out, d)
        single = []
        for v in range(nvec):     # the same plan, one vector at a time
            o1 = torch.zeros(out_len, dtype=getattr(torch, cname), device=DEV)
            dv = torch.from_numpy(np.ascontiguousarray(data[v], dtype=cdt)).to(DEV)
            if ttype == 1:
                plan.execute(dv, o1)
            else:
                plan.execute(o1, dv)
            single.append(o1.cpu().numpy())
        info = plan.info()
        torch.cuda.synchronize()
    got = out if host else out.cpu().numpy()
    return got, np.stack(single), info


CASES = [
    # dim, N, dt, eps, opts
    (1, (1500,), "f32", 1e-5, {}),
    (1, (1500,), "f64", 1e-12, {}),
    (2, (100, 70), "f32", 1e-5, {}),
    (2, (100, 70), "f64", 1e-9, {}),
    (2, (100, 70), "f32", 1e-6, {"method": nf.METHOD_SM}),
    (2, (100, 70), "f32", 1e-3, {"method": nf.METHOD_GM_SORT}),
    (2, (100, 70), "f64", 1e-6, {"method": nf.METHOD_GM}),
    (2, (100, 70), "f32", 1e-5, {"regtile_cols": 2}),
    (3, (20, 24, 36), "f32", 1e-6, {}),
    (3, (20, 24, 36), "f32", 1e-6, {"igroup": 1}),
    (3, (20, 24, 36), "f64", 1e-12, {}),
    (3, (20, 24, 36), "f32", 1e-4, {"method": nf.METHOD_SM}),
    (3, (20, 24, 36), "f64", 1e-9, {"method": nf.METHOD_GM}),
]


@pytest.mark.parametrize("ttype", [1, 2])
@pytest.mark.parametrize("dim,N,dt,eps,opts", CASES)
def test_batch_matches_oracle(dim, N, dt, eps, opts, ttype):
    """5 vectors in passes of 2, 2 and 1 (a batched cuFFT plan of each size)."""
    rng = np.random.default_rng(40 + dim)
    M = 12000
    nvec = 5
    pts = _pts(dim, M, "uniform", rng, dt)
    n_in = M if ttype == 1 else int(np.prod(N))
    data = np.stack([_cplx(n_in, rng, dt) for _ in range(nvec)])
    iflag = -1 if ttype == 1 else 1
    got, single, info = _run_batch(ttype, pts, data, N, eps, iflag, dt, nvec, dict(opts, batch=2))
    assert info["batch"] == 2
    for v in range(nvec):
        if ttype == 1:
            ref = oracle.nufft_type1(pts, data[v], N, eps, iflag).ravel()
        else:
            ref = oracle.nufft_type2(pts, data[v], N, eps, iflag)
        assert oracle.rel_l2(got[v], ref) <= TOL_O2[dt], f"vector {v}"
        assert oracle.rel_l2(got[v], single[v]) <= SAME[dt], f"vector {v} vs single execute"


def test_batch_host_pointers_and_default_pass():
    """Host arrays through the staging buffers; default pass = as many fine
    grids as fit in 1 GiB, at most 64 (here all 7 vectors in one pass)."""
    rng = np.random.default_rng(7)
    N = (64, 48)
    M = 5000
    dt = "f32"
    pts = _pts(2, M, "uniform", rng, dt)
    data = np.stack([_cplx(M, rng, dt) for _ in range(7)])
    got, single, info = _run_batch(1, pts, data, N, 1e-5, 1, dt, 7, {}, host=True)
    cells = info["n1"] * info["n2"]
    assert info["batch"] == max(1, min(64, (1 << 30) // (cells * 8)))
    for v in range(7):
        ref = oracle.nufft_type1(pts, data[v], N, 1e-5, 1).ravel()
        assert oracle.rel_l2(got[v], ref) <= TOL_O2[dt]
        assert oracle.rel_l2(got[v], single[v]) <= SAME[dt]
    # type 2, host arrays, passes of 3 (3, 3, 1)
    fk = np.stack([_cplx(int(np.prod(N)), rng, dt) for _ in range(7)])
    got2, single2, _ = _run_batch(2, pts, fk, N, 1e-5, -1, dt, 7, {"batch": 3}, host=True)
    for v in range(7):
        ref = oracle.nufft_type2(pts, fk[v], N, 1e-5, -1)
        assert oracle.rel_l2(got2[v], ref) <= TOL_O2[dt]
        assert oracle.rel_l2(got2[v], single2[v]) <= SAME[dt]


def test_batch_edge_cases():
    rng = np.random.default_rng(8)
    N = (32, 20)
    pts = [torch.from_numpy(p).to(DEV) for p in _pts(2, 300, "uniform", rng, "f32")]
    with nf.Plan(1, N, -1, 1e-5, "complex64") as plan:
        with pytest.raises(nf.NufftError) as ei:   # no points yet
            plan.execute_batch(2, torch.zeros(600, dtype=torch.complex64, device=DEV),
                               torch.zeros(2 * 640, dtype=torch.complex64, device=DEV))
        assert ei.value.code == nf.ERR_NO_POINTS
        plan.setpts(*pts)
        f = torch.full((640,), 3 + 1j, dtype=torch.complex64, device=DEV)
        plan.execute_batch(0, None, f)             # nothing happens
        torch.cuda.synchronize()
        assert torch.all(f == 3 + 1j)
        with pytest.raises(nf.NufftError) as ei:
            plan.execute_batch(-1, None, f)
        assert ei.value.code == nf.ERR_BAD_ARG
        with pytest.raises(nf.NufftError) as ei:
            plan.set_opt("batch", 1025)
        assert ei.value.code == nf.ERR_BAD_OPT
        # after a single execute the plan grows its fine grids for a pass of 4
        c = torch.from_numpy(_cplx(4 * 300, rng, "f32")).to(DEV)
        out = torch.zeros(4 * 640, dtype=torch.complex64, device=DEV)
        plan.execute(c[:300], out[:640])
        one = out[:640].cpu().numpy().copy()
        plan.set_opt("batch", 4)
        plan.execute_batch(4, c, out)
        t = plan.timings()
        torch.cuda.synchronize()
        assert oracle.rel_l2(out[:640].cpu().numpy(), one) <= SAME["f32"]
        assert t["exec"] >= t["spread_interp"] > 0 and t["fft"] > 0


def test_batch_zero_points():
    """M = 0: type 1 gives zeros for every vector, type 2 writes nothing."""
    with nf.Plan(1, (16, 8), -1, 1e-5, "complex64") as plan:
        plan.setpts(torch.zeros(0, device=DEV), torch.zeros(0, device=DEV))
        f = torch.full((3, 128), 5.0, dtype=torch.complex64, device=DEV)
        plan.execute_batch(3, None, f)
        torch.cuda.synchronize()
        assert torch.all(f == 0)
