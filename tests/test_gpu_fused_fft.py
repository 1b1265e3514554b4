"""The fused, pruned fine-grid FFT of 2D complex64 plans (power-of-two fine
grids from 256 to 4096), against the oracle's three-step NUFFT and the direct
sums of eq. (1) / (3) of "cuFINUFFT: a load-balanced GPU library for
general-purpose nonuniform FFTs", and against the same plan run through cuFFT
and the separate correction kernels (option "fft" = 1).

Tolerances as in the other parity tests: 1e-5 relative l2 against the oracle's
NUFFT (only rounding differs); against the direct sums at most 2 eps, or 25 %
above the oracle NUFFT's own error on the same outputs where that is larger
(a few sampled modes at the edges of I_N, where the correction factors are
largest, can sit above 2 eps).  Between the two FFT paths only the
single-precision rounding of the FFT differs: 1e-6.
"""
import numpy as np
import pytest
import torch

import nonuniform_fft_gb300 as nf
import oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

# N -> fine grid n = smallest 2^a 3^b 5^c >= 2 N: (128, 128) -> (256, 256);
# odd (127, 255) -> (256, 512); (1024, 128) -> (2048, 256);
# (2048, 128) -> (4096, 256); (64, 64) -> (128, 128); (64, 1024) -> (128, 2048)
SIZES = [(128, 128), (127, 255), (1024, 128), (2048, 128), (64, 64), (64, 1024)]


def _pts(M, rng):
    return [rng.uniform(-np.pi, np.pi, M).astype(np.float32) for _ in range(2)]


def _cplx(n, rng):
    return (rng.standard_normal(n) + 1j * rng.standard_normal(n)).astype(np.complex64)


def _check_direct(got, o2, ref, eps):
    err, err_o2 = oracle.rel_l2(got, ref), oracle.rel_l2(o2, ref)
    assert err <= max(2 * eps, 1.25 * err_o2), f"vs direct {err:.3e} (oracle NUFFT {err_o2:.3e})"


def _run(ttype, N, pts, data, eps, iflag, opts=None, nvec=1):
    xs = [torch.from_numpy(p).to(DEV) for p in pts]
    d = torch.from_numpy(data).to(DEV)
    M = len(pts[0])
    out = torch.zeros(nvec * (int(np.prod(N)) if ttype == 1 else M), dtype=torch.complex64, device=DEV)
    with nf.Plan(ttype, N, iflag, eps, "complex64", **(opts or {})) as plan:
        plan.setpts(*xs)
        if ttype == 1:
            plan.execute_batch(nvec, d, out) if nvec > 1 else plan.execute(d, out)
        else:
            plan.execute_batch(nvec, out, d) if nvec > 1 else plan.execute(out, d)
        info = plan.info()
        torch.cuda.synchronize()
    return out.cpu().numpy(), info


@pytest.mark.parametrize("N", SIZES)
@pytest.mark.parametrize("eps", [1e-2, 1e-5])
def test_fused_type1_matches_oracle(N, eps):
    rng = np.random.default_rng(61)
    M = 20000
    pts = _pts(M, rng)
    c = _cplx(M, rng)
    for iflag in (-1, 1):
        f, info = _run(1, N, pts, c, eps, iflag)
        assert info["fft"] == 1 and info["n1"] & (info["n1"] - 1) == 0
        f = f.reshape(N[1], N[0])
        o2 = oracle.nufft_type1(pts, c, N, eps, iflag)
        assert oracle.rel_l2(f, o2) <= 1e-5
        ks = [np.array([-(n // 2), -1, 0, 1, n - n // 2 - 1]) for n in N]
        ref = oracle.direct_type1(pts, c, N, iflag, modes=ks)
        sel = np.ix_(*[k + n // 2 for k, n in zip(reversed(ks), reversed(N))])
        _check_direct(f[sel], o2[sel], ref, eps)


@pytest.mark.parametrize("N", SIZES)
@pytest.mark.parametrize("eps", [1e-2, 1e-5])
def test_fused_type2_matches_oracle(N, eps):
    rng = np.random.default_rng(62)
    M = 20000
    pts = _pts(M, rng)
    fk = _cplx(int(np.prod(N)), rng)
    for iflag in (-1, 1):
        c, info = _run(2, N, pts, fk, eps, iflag)
        assert info["fft"] == 1
        o2 = oracle.nufft_type2(pts, fk, N, eps, iflag)
        assert oracle.rel_l2(c, o2) <= 1e-5
        tg = np.arange(0, M, 97)
        ref = oracle.direct_type2(pts, fk, N, iflag, targets=tg)
        _check_direct(c[tg], o2[tg], ref, eps)


@pytest.mark.parametrize("ttype", [1, 2])
@pytest.mark.parametrize("N", [(127, 255), (1024, 128)])
def test_fused_matches_cufft_path(ttype, N):
    rng = np.random.default_rng(63)
    M = 50000
    pts = _pts(M, rng)
    data = _cplx(M if ttype == 1 else int(np.prod(N)), rng)
    a, ia = _run(ttype, N, pts, data, 1e-6, 1)
    b, ib = _run(ttype, N, pts, data, 1e-6, 1, {"fft": 1})
    assert ia["fft"] == 1 and ib["fft"] == 0
    assert oracle.rel_l2(a, b) <= 1e-6


@pytest.mark.parametrize("ttype", [1, 2])
def test_fused_batched(ttype):
    """Three vectors in one pass and in passes of two: each equals its own
    single-vector execute."""
    rng = np.random.default_rng(64)
    N, M, nvec = (128, 128), 8000, 3
    pts = _pts(M, rng)
    size = M if ttype == 1 else int(np.prod(N))
    data = _cplx(nvec * size, rng)
    outs = [_run(ttype, N, pts, data, 1e-5, -1, {"batch": b}, nvec=nvec)[0] for b in (0, 2)]
    per = np.concatenate([_run(ttype, N, pts, data[v * size:(v + 1) * size], 1e-5, -1)[0]
                          for v in range(nvec)])
    for o in outs:
        assert oracle.rel_l2(o, per) <= 1e-6


def test_fused_not_used_where_unsupported():
    """Non-power-of-two or small fine grids and complex128 plans keep cuFFT."""
    rng = np.random.default_rng(65)
    pts = _pts(1000, rng)
    c = _cplx(1000, rng)
    for N in [(100, 70), (32, 32)]:   # fine grids 200 x 140 (not 2^a) and 64 x 64 (below 128)
        _, info = _run(1, N, pts, c, 1e-5, -1)
        assert info["fft"] == 0
    xs = [torch.from_numpy(p.astype(np.float64)).to(DEV) for p in pts]
    with nf.Plan(1, (128, 128), -1, 1e-9, "complex128") as plan:
        plan.setpts(*xs)
        assert plan.info()["fft"] == 0


def test_fused_repeated_executes_on_one_plan():
    """The fused x pass leaves the fine grids it read zeroed, and the next type
    1 execute skips the clear: executes on one plan (one vector, a batch of two
    that grows the plan's grids, one vector, a batch of two) each equal a fresh
    plan's result."""
    rng = np.random.default_rng(66)
    N, M = (128, 256), 6000
    pts = _pts(M, rng)
    cs = [_cplx(M, rng) for _ in range(6)]
    xs = [torch.from_numpy(p).to(DEV) for p in pts]
    nm = int(np.prod(N))
    got = []
    with nf.Plan(1, N, -1, 1e-5, "complex64") as plan:
        plan.setpts(*xs)
        assert plan.info()["fft"] == 1
        for group in ([0], [1, 2], [3], [4, 5]):
            c = torch.from_numpy(np.concatenate([cs[i] for i in group])).to(DEV)
            f = torch.zeros(len(group) * nm, dtype=torch.complex64, device=DEV)
            if len(group) == 1:
                plan.execute(c, f)
            else:
                plan.execute_batch(len(group), c, f)
            got += list(f.cpu().numpy().reshape(len(group), nm))
    for i in range(6):
        ref, _ = _run(1, N, pts, cs[i], 1e-5, -1)
        assert oracle.rel_l2(got[i], ref) <= 1e-6, i
