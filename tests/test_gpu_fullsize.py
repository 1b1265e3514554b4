"""The five benchmark workloads at full size, in the default launch
configuration that bench.py times, checked against the oracle.

Outputs the oracle can compute one by one: type 1 on a tensor grid of modes
drawn uniformly from I_N (plus k = 0), type 2 at randomly drawn targets, both
by the direct sums of eq. (1) / (3) of "cuFINUFFT: a load-balanced GPU library
for general-purpose nonuniform FFTs".  Bound: 2 eps, except the 3D double
precision eps = 1e-12 workload, where the method itself (the oracle's own
three-step NUFFT in double precision) reaches about 3 eps, so 4 eps.  Every
workload is also compared over its whole output array (every mode for type 1,
every point for type 2) with the oracle's three-step NUFFT at the same w, beta
and fine grid: 1e-5 relative l2 for complex64, 1e-12 for complex128.  The
oracle runs on all host cores, which keeps the 3D workloads (3.2e7 points at
w = 7, 1e7 points at w = 13) to tens of seconds each.
"""
import numpy as np
import pytest
import torch

import nonuniform_fft_gb300 as nf
import oracle
from nonuniform_fft_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BOUND = {"2d_t1_f32_N64_M1e4": 2, "2d_f32_N1024_M1e7": 2, "2d_t1_f32_N1024_M1e7_cluster": 2,
         "3d_f32_N128_M3.2e7": 2, "3d_f64_N64_M1e7_mix": 4, "1d_f64_N1e6_M1e7": 2}
TOL_O2 = {"f32": 1e-5, "f64": 1e-12}


def _run(wl, t, pts, data):
    cname = "complex64" if wl.dtype == "f32" else "complex128"
    xs = [torch.from_numpy(p).to(DEV) for p in pts]
    d = torch.from_numpy(data).to(DEV)
    out = torch.empty(int(np.prod(wl.N)) if t == 1 else wl.M, dtype=getattr(torch, cname), device=DEV)
    with nf.Plan(t, wl.N, wl.iflag[t], wl.eps, cname) as plan:
        plan.setpts(*xs)
        if t == 1:
            plan.execute(d, out)
        else:
            plan.execute(out, d)
        torch.cuda.synchronize()
    return out.cpu().numpy()


def _sample_modes(N, k, rng):
    ks = []
    for n in N:
        kk = rng.choice(np.arange(-(n // 2), n - n // 2), size=min(k, n), replace=False)
        ks.append(np.unique(np.concatenate([kk, [0]])))
    return ks


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_type1_full_size(name):
    wl = W.WORKLOADS[name]
    pts, c = W.sample(wl)
    f = _run(wl, 1, pts, c).reshape(tuple(reversed(wl.N)))
    rng = np.random.default_rng(100)
    ks = _sample_modes(wl.N, {1: 64, 2: 14, 3: 7}[wl.dim], rng)
    ref = oracle.direct_type1(pts, c, wl.N, wl.iflag[1], modes=ks)
    got = f[np.ix_(*[k + n // 2 for k, n in zip(reversed(ks), reversed(wl.N))])]
    err = oracle.rel_l2(got, ref)
    assert err <= BOUND[name] * wl.eps, f"{name}: type 1 vs direct sum {err:.3e}"
    o2 = oracle.nufft_type1(pts, c, wl.N, wl.eps, wl.iflag[1])
    e2 = oracle.rel_l2(f, o2)
    assert e2 <= TOL_O2[wl.dtype], f"{name}: type 1 vs the oracle's NUFFT {e2:.3e}"


@pytest.mark.parametrize("name", [n for n, w in W.WORKLOADS.items() if 2 in w.types])
def test_type2_full_size(name):
    wl = W.WORKLOADS[name]
    pts, _ = W.sample(wl)
    fk = W.coefficients(wl)
    c = _run(wl, 2, pts, fk)
    rng = np.random.default_rng(101)
    tg = rng.choice(wl.M, size=120, replace=False)
    ref = oracle.direct_type2(pts, fk, wl.N, wl.iflag[2], targets=tg)
    err = oracle.rel_l2(c[tg], ref)
    assert err <= BOUND[name] * wl.eps, f"{name}: type 2 vs direct sum {err:.3e}"
    o2 = oracle.nufft_type2(pts, fk, wl.N, wl.eps, wl.iflag[2])
    e2 = oracle.rel_l2(c, o2)
    assert e2 <= TOL_O2[wl.dtype], f"{name}: type 2 vs the oracle's NUFFT {e2:.3e}"
