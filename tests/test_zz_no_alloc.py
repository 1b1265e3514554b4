"""The no-allocation bin sort (nufft_binsort_noalloc) against the plan path.

It is for callers that cannot allocate device memory (under a host-owned
memory pool, in real-time loops), so its scratch is a fixed array inside the
library.  This file is collected last: a failure
here leaves every other test already run.  It must pass alone in a fresh
process and after the other tests (the shared scratch keeps the previous
call's contents).
"""
import ctypes

import numpy as np
import pytest
import torch

import nonuniform_fft_gb300 as nf

DEV = torch.device("cuda:0")


def _lib():
    lib = nf.load_library()
    f = lib.nufft_binsort_noalloc
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [ctypes.c_int, ctypes.c_int, I64, P, P, P, ctypes.POINTER(I64),
                  ctypes.POINTER(I64), P, P, P]
    f.restype = ctypes.c_int
    return f


def _points(dim, M, seed, dtype):
    rng = np.random.default_rng(seed)
    pts = [rng.uniform(-np.pi, np.pi, M) for _ in range(dim)]
    pts[0][: M // 3] = np.mod(rng.normal(0, 0.2, M // 3) + np.pi, 2 * np.pi) - np.pi  # a cluster
    return [torch.from_numpy(p.astype(dtype)).to(DEV) for p in pts]


def _plan_sort(dim, N, xs, bins, cname):
    opts = {f"bin{i + 1}": b for i, b in enumerate(bins)}
    with nf.Plan(1, N, -1, 1e-6, cname, **opts) as plan:
        plan.setpts(*xs)
        info = plan.info()
        ref = plan.sort()
    n = [info["n1"], info["n2"], info["n3"]][:dim]
    m = [info["bin1"], info["bin2"], info["bin3"]][:dim]
    return n, m, ref


def _noalloc_sort(f, dim, dtype_code, xs, n, m, nbins):
    M = xs[0].numel()
    counts = torch.full((nbins,), -7, dtype=torch.int32, device=DEV)
    perm = torch.full((max(M, 1),), -7, dtype=torch.int32, device=DEV)
    na = (ctypes.c_int64 * dim)(*n)
    ma = (ctypes.c_int64 * dim)(*m)
    stream = torch.cuda.current_stream().cuda_stream
    rc = f(dim, dtype_code, M, xs[0].data_ptr(), xs[1].data_ptr(),
           xs[2].data_ptr() if dim == 3 else None, na, ma, counts.data_ptr(), perm.data_ptr(),
           stream)
    return rc, counts.cpu().numpy(), perm[:M].cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("dim,N,bins,dt", [(2, (300, 200), (32, 16), "f32"),
                                           (3, (40, 24, 36), (8, 8, 4), "f64")])
def test_noalloc_binsort_matches_plan_twice(dim, N, bins, dt):
    f = _lib()
    cname, rdt, code = ("complex64", np.float32, 0) if dt == "f32" else ("complex128", np.float64, 1)
    for call, (M, seed) in enumerate([(200_000, 1), (150_000, 2)]):   # two calls in a row
        xs = _points(dim, M, seed, rdt)
        n, m, ref = _plan_sort(dim, N, xs, bins, cname)
        rc, counts, perm = _noalloc_sort(f, dim, code, xs, n, m, ref["counts"].size)
        assert rc == nf.OK, nf.strerror(rc)
        np.testing.assert_array_equal(counts, ref["counts"])
        for lo, cnt in zip(ref["starts"], ref["counts"]):
            np.testing.assert_array_equal(np.sort(perm[lo:lo + cnt]), np.sort(ref["perm"][lo:lo + cnt]))


@pytest.mark.gpu
def test_noalloc_binsort_rejects_sizes_beyond_limit():
    f = _lib()
    x = torch.zeros(16, dtype=torch.float32, device=DEV)
    counts = torch.zeros(16, dtype=torch.int32, device=DEV)
    n = (ctypes.c_int64 * 2)(64, 64)
    m = (ctypes.c_int64 * 2)(16, 16)
    rc = f(2, 0, (1 << 20) + 1, x.data_ptr(), x.data_ptr(), None, n, m, counts.data_ptr(),
           counts.data_ptr(), None)
    assert rc == nf.ERR_TOO_LARGE
    big = (ctypes.c_int64 * 2)(1 << 20, 1 << 20)
    one = (ctypes.c_int64 * 2)(1, 1)
    rc = f(2, 0, 16, x.data_ptr(), x.data_ptr(), None, big, one, counts.data_ptr(),
           counts.data_ptr(), None)
    assert rc == nf.ERR_TOO_LARGE


@pytest.mark.parametrize("n3", [16, 8])
def test_noalloc_binsort_bin_count_overflow_is_rejected(n3):
    """Bin counts whose product overflows int64 (2^30 * 2^30 * n3 single-cell
    bins wraps to 0 or to a negative number) must give TOO_LARGE from the
    argument checks, which run before any CUDA call, so no GPU is needed."""
    f = _lib()
    buf = (ctypes.c_int32 * 16)()
    ptr = ctypes.addressof(buf)
    n = (ctypes.c_int64 * 3)(1 << 30, 1 << 30, n3)
    one = (ctypes.c_int64 * 3)(1, 1, 1)
    rc = f(3, 0, 16, ptr, ptr, ptr, n, one, ptr, ptr, None)
    assert rc == nf.ERR_TOO_LARGE
