"""The single-precision fold of setpts against the double-precision fold.

setpts folds each coordinate to its fine-grid cell (g = n frac(x / 2 pi),
node l at l h, "cuFINUFFT: a load-balanced GPU library for general-purpose
nonuniform FFTs", eq. (7)).  The cell must equal the oracle's, which folds in
double precision.  For single-precision coordinates the library first tries a
fold in float arithmetic only (the double constant 1/(2 pi) split exactly into
three floats, exact products by fused multiply-add, an error bound) and falls
back to the double fold when the result is within its bound of a cell
boundary.  This test restates that float computation in numpy (float32
operations are IEEE single precision; a fused multiply-add x c - p is exact
in float64 and then rounded once) and checks, on random and on adversarial
coordinates -- the floats nearest every cell boundary -- that wherever it
answers, its cell is the double fold's.  The GPU parity tests check the
kernel's integer results against the oracle.
"""
import numpy as np
import pytest

import oracle

F = np.float32
C = 1.0 / (2.0 * np.pi)   # the double constant both folds use


def _split3():
    c0 = F(C)
    r = C - float(c0)
    c1 = F(r)
    c2 = F(r - float(c1))
    assert (float(c0) + float(c1)) + float(c2) == C
    return c0, c1, c2


def _fma(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(F)


def _two_sum(a, b):
    s = (a + b).astype(F)
    bv = (s - a).astype(F)
    lo = ((a - (s - bv)) + (b - bv)).astype(F)
    return s, lo


def fold_fast(x, n):
    """(ok, cell) of the float fold for float32 x and grid size n."""
    x = x.astype(F)
    c0, c1, c2 = (np.full_like(x, v) for v in _split3())
    p0 = (x * c0).astype(F)
    e0 = _fma(x, c0, -p0)
    p1 = (x * c1).astype(F)
    e1 = _fma(x, c1, -p1)
    p2 = (x * c2).astype(F)
    f, fl = _two_sum(p0, (-np.floor(p0)).astype(F))
    tail = (((e0 + p1) + (e1 + p2)) + fl).astype(F)
    s, sl = _two_sum(f, tail)
    neg, big = s < 0, s >= 1
    t, tl = _two_sum(s, np.where(neg, F(1), F(-1)).astype(F))
    fix = neg | big
    s = np.where(fix, t, s).astype(F)
    sl = np.where(fix, (sl + tl).astype(F), sl).astype(F)
    nf = F(n)
    h = (s * nf).astype(F)
    l = (_fma(s, np.full_like(s, nf), -h) + (sl * nf).astype(F)).astype(F)
    r = np.rint(h).astype(F)
    d = ((h - r) + l).astype(F)
    delta = (nf * (np.abs(p0) + F(1)) * F(5.6843419e-14)).astype(F)
    k = r.astype(np.int64) - (d < 0)
    ok = (np.abs(x) <= 1024) & (np.abs(d) > delta) & (k >= 0) & (k < n)
    return ok, k


def cell_double(x, n):
    """The double fold, operation by operation (IEEE double in numpy)."""
    t = x.astype(np.float64) * C
    t = t - np.floor(t)
    g = t * float(n)
    g = np.where(g >= n, g - n, g)
    return np.floor(g).astype(np.int64)


def test_double_fold_restatement_matches_oracle():
    rng = np.random.default_rng(0)
    x = rng.uniform(-40, 40, 2000).astype(F)
    for n in (128, 2048, 1280, 2_000_000):
        ref = np.array([int(np.floor(oracle.grid_coord(float(v), n))) for v in x])
        np.testing.assert_array_equal(cell_double(x, n), ref)


def _boundary_floats(n, per_side=3):
    """The float32 values nearest the coordinates of cell boundaries k h
    (and of the same boundaries one and two periods away)."""
    k = np.arange(n + 1, dtype=np.float64)
    out = []
    for shift in (0.0, -2 * np.pi, 2 * np.pi, 4 * np.pi):
        b = (2 * np.pi * k / n + shift).astype(F)
        v = b.copy()
        out.append(v)
        lo, hi = v.copy(), v.copy()
        for _ in range(per_side):
            lo = np.nextafter(lo, F(-np.inf))
            hi = np.nextafter(hi, F(np.inf))
            out += [lo.copy(), hi.copy()]
    return np.concatenate(out)


@pytest.mark.parametrize("n", [128, 256, 2048, 4096, 1280, 1_000_003, 2_000_000])
def test_float_fold_cells_equal_double_fold(n):
    rng = np.random.default_rng(n)
    xs = [rng.uniform(-np.pi, np.pi, 2_000_000).astype(F),
          rng.uniform(-1024, 1024, 200_000).astype(F),
          np.array([0.0, -0.0, np.pi, -np.pi, 2 * np.pi, 1024, -1024], dtype=F)]
    if n <= 4096:
        xs.append(_boundary_floats(n))
    else:
        idx = rng.choice(n + 1, 200_000, replace=False).astype(np.float64)
        b = (2 * np.pi * idx / n).astype(F)
        xs += [b, np.nextafter(b, F(-np.inf)), np.nextafter(b, F(np.inf))]
    x = np.concatenate(xs)
    ok, k = fold_fast(x, n)
    ref = cell_double(x, n)
    bad = ok & (k != ref)
    assert not bad.any(), f"n={n}: {bad.sum()} cells differ, e.g. x={x[bad][:5]}"
    # random coordinates almost never need the double fold
    okr, _ = fold_fast(xs[0], n)
    assert okr.mean() > 0.9999
