"""Accuracy of the two-float (double-single) ES kernel used by the
double-precision kernels, "cuFINUFFT: a load-balanced GPU library for
general-purpose nonuniform FFTs" eq. (5), phi(z) = exp(beta (sqrt(1-z^2)-1)).
The library header is compiled as host code (contraction off) and compared
with a 40-digit evaluation by Python's decimal module."""
import os
import shutil
import subprocess
from decimal import Decimal, getcontext

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("df64") / "drv")
    subprocess.run([nvcc, "-O2", "-std=c++17", "-Xcompiler", "-ffp-contract=off",
                    os.path.join(HERE, "host", "df64_es_driver.cu"), "-o", exe],
                   check=True, capture_output=True)
    return exe


def _exact(z, beta):
    getcontext().prec = 40
    zd, bd = Decimal(z), Decimal(beta)
    return float((bd * ((1 - zd * zd).sqrt() - 1)).exp())


def test_df64_es_kernel_accuracy(driver):
    rng = np.random.default_rng(3)
    cases = []
    for w in range(2, 17):
        beta = 2.30 * w
        zs = np.concatenate([[-1.0, 1.0, 0.0, 1e-9, -0.5, 0.999999999, -0.9999], rng.uniform(-1, 1, 60)])
        cases += [(float(z), beta) for z in zs]
    for sigma in (1.25, 1.5):        # the sigma < 2 shapes
        for w in (5, 9, 16):
            beta = 2.30 * w * (4 / 3) * (1 - 0.5 / sigma)
            cases += [(float(z), beta) for z in rng.uniform(-1, 1, 20)]
    inp = "".join(f"{z!r} {b!r}\n" for z, b in cases)
    out = subprocess.run([driver], input=inp, capture_output=True, text=True, check=True).stdout
    rows = [[float(v) for v in line.split()] for line in out.strip().splitlines()]
    assert len(rows) == len(cases)
    # absolute error, i.e. relative to the kernel's peak phi(0) = 1: that is
    # the error a weighted sum sees.  A double-precision evaluation of the
    # same formula is off by up to about beta * 1e-16 * phi (~4e-15); the
    # two-float one carries 48 bits and stays below 8e-15, with the series
    # exponential and with the table one (2^(j/64) and a degree-6 series).
    for (z, beta), (sh, sl, th, tl) in zip(cases, rows):
        ref = _exact(z, beta)
        assert abs((sh + sl) - ref) <= 8e-15, (z, beta, sh + sl, ref)
        assert abs((th + tl) - ref) <= 8e-15, ("table", z, beta, th + tl, ref)


@pytest.fixture(scope="module")
def dot_driver(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("df64dot") / "drv")
    subprocess.run([nvcc, "-O2", "-std=c++17", "-Xcompiler", "-ffp-contract=off",
                    os.path.join(HERE, "host", "df64_dot_driver.cu"), "-o", exe],
                   check=True, capture_output=True)
    return exe


def test_df64_lazy_dot_products(dot_driver):
    """Row sums of the double-precision interpolator: up to 16 products of
    two-floats, accumulated without renormalisation in two chains and
    renormalised once, against the exact sum of the same two-float products
    (Fraction arithmetic).  The bound is relative to the sum of |terms|: two
    two-float roundings per product (2^-47 each) plus the deferred float
    rounding of the low parts.  The renormalising form df_fma is held to the
    same bound."""
    from fractions import Fraction

    def split(x):
        hi = float(np.float32(x))
        lo = float(np.float32(x - hi))
        return hi, lo

    rng = np.random.default_rng(7)
    lines, cases = [], []
    for n in list(range(1, 17)) * 12:
        kind = rng.integers(0, 3)
        a = rng.standard_normal(n) * (10.0 ** rng.uniform(-3, 3, n) if kind == 2 else 1.0)
        b = np.abs(rng.uniform(0, 1, n)) if kind != 1 else rng.standard_normal(n)
        if kind == 1 and n > 1:              # heavy cancellation
            a[-1] = -sum(a[:-1] * b[:-1]) / b[-1]
        lines.append(f"{n} " + " ".join(f"{float(x)!r} {float(y)!r}" for x, y in zip(a, b)))
        cases.append((a, b))
    out = subprocess.run([dot_driver], input="\n".join(lines) + "\n", capture_output=True, text=True,
                         check=True).stdout.strip().splitlines()
    assert len(out) == len(cases)
    for (a, b), line in zip(cases, out):
        lh, ll, sh, sl = (float(v) for v in line.split())
        exact = Fraction(0)
        mag = Fraction(0)
        for x, y in zip(a, b):
            xh, xl = split(x)
            yh, yl = split(y)
            t = (Fraction(xh) + Fraction(xl)) * (Fraction(yh) + Fraction(yl))
            exact += t
            mag += abs(t)
        bound = float(mag) * 2.0 ** -44
        assert abs(float(Fraction(lh) + Fraction(ll) - exact)) <= bound, (len(a), lh, ll, float(exact))
        assert abs(float(Fraction(sh) + Fraction(sl) - exact)) <= bound, (len(a), sh, sl, float(exact))
