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


def _fold_hl(x, n):
    """The float fold's g = h + l and its error bound delta (eligible where
    |x| <= 1024)."""
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
    delta = (nf * (np.abs(p0) + F(1)) * F(5.6843419e-14)).astype(F)
    return np.abs(x) <= 1024, h, l, delta


def fold_fast(x, n):
    """(ok, cell) of the float fold for float32 x and grid size n."""
    elig, h, l, delta = _fold_hl(x, n)
    r = np.rint(h).astype(F)
    d = ((h - r) + l).astype(F)
    k = r.astype(np.int64) - (d < 0)
    ok = elig & (np.abs(d) > delta) & (k >= 0) & (k < n)
    return ok, k


def node_fast(x, n, oc):
    """(ok, node) of the float fold's window-origin node ceil(g - oc), oc =
    1/2 (odd w) or 0 (even w), taken mod n."""
    elig, h, l, delta = _fold_hl(x, n)
    h2 = (h - F(oc)).astype(F)
    r = np.rint(h2).astype(F)
    d = ((h2 - r) + l).astype(F)
    k = r.astype(np.int64) + (d > 0)
    ok = elig & (np.abs(d) > delta) & (k >= 0) & (k <= n) & ((oc == 0) | (n <= 1 << 22))
    return ok, np.where(k == n, 0, k)


def cell_double(x, n):
    """The double fold, operation by operation (IEEE double in numpy)."""
    t = x.astype(np.float64) * C
    t = t - np.floor(t)
    g = t * float(n)
    g = np.where(g >= n, g - n, g)
    return np.floor(g).astype(np.int64)


def node_double(x, n, w):
    """The oracle's bin index by window origin, ceil(g - w/2) + floor(w/2) =
    ceil(g - oc) (mod n), from the double fold."""
    t = x.astype(np.float64) * C
    t = t - np.floor(t)
    g = t * float(n)
    g = np.where(g >= n, g - n, g)
    return np.mod(np.ceil(g - (0.5 * w - w // 2)).astype(np.int64), n)


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


def _half_boundary_floats(n, per_side=3):
    """The float32 values nearest the coordinates 2 pi (k + 1/2) / n (the
    origin boundaries of odd w), and one period either side."""
    k = np.arange(n + 1, dtype=np.float64) + 0.5
    out = []
    for shift in (0.0, -2 * np.pi, 2 * np.pi):
        v = (2 * np.pi * k / n + shift).astype(F)
        out.append(v)
        lo, hi = v.copy(), v.copy()
        for _ in range(per_side):
            lo = np.nextafter(lo, F(-np.inf))
            hi = np.nextafter(hi, F(np.inf))
            out += [lo.copy(), hi.copy()]
    return np.concatenate(out)


@pytest.mark.parametrize("w", [7, 6, 3, 8])
@pytest.mark.parametrize("n", [128, 256, 2048, 1280])
def test_float_fold_origins_equal_double_fold(n, w):
    """setpts bins the slab spreader's points by window origin: the node
    ceil(g - oc) (oc = 1/2 for odd w, 0 for even w) from the float fold,
    where it answers, equals the double fold's ceil(g - w/2) + floor(w/2)
    (mod n), on random coordinates and on the floats nearest the origin
    boundaries (half-integer g for odd w, integer g for even w)."""
    rng = np.random.default_rng(n + w)
    oc = 0.5 if w % 2 else 0.0
    x = np.concatenate([rng.uniform(-np.pi, np.pi, 1_000_000).astype(F),
                        rng.uniform(-1024, 1024, 100_000).astype(F),
                        _half_boundary_floats(n) if w % 2 else _boundary_floats(n),
                        np.array([0.0, -0.0, np.pi, -np.pi, 2 * np.pi], dtype=F)])
    ok, k = node_fast(x, n, oc)
    ref = node_double(x, n, w)
    bad = ok & (k != ref)
    assert not bad.any(), f"n={n} w={w}: {bad.sum()} origins differ, e.g. x={x[bad][:5]}"
    assert ok[:1_000_000].mean() > 0.9999
