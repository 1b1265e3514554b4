"""Seeded synthetic workloads for the nonuniform FFT.

Random inputs only: this module holds none of the transform's arithmetic, so
that the CUDA path and the CPU oracle can be fed identical inputs without
sharing code.

Point distributions follow the two extremes the cuFINUFFT paper benchmarks
(Sec. IV, "Tasks"): "rand" (iid uniform over the periodic box [-pi, pi)^d) and
clustered points.  The clustered variant here is iid normal(0, sigma) per
coordinate, wrapped into [-pi, pi).  Strengths c_j (type 1) and coefficients
f_k (type 2) have iid standard normal real and imaginary parts.

Recipe (numpy PCG64 via ``default_rng(seed)``, draws in float64, then cast to
the plan's real type): x, then y, (then z); then Re, Im of the strengths.
The type 2 coefficients use ``seed + 100``.  A "mix" workload draws its first
M/2 points uniform and the last M/2 clustered, then shuffles them once with
the same generator.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np

TWO_PI = 2.0 * np.pi


@dataclass(frozen=True)
class Workload:
    name: str
    dim: int
    N: tuple            # modes per dimension (N1, N2[, N3])
    M: int              # number of nonuniform points
    eps: float
    dtype: str          # "f32" (complex64) or "f64" (complex128)
    types: tuple        # transform types exercised (1, 2)
    dist: str           # "uniform" | "cluster" | "mix"
    sigma: float = 0.0  # normal width for clustered points
    seed: int = 0
    iflag: dict = field(default_factory=lambda: {1: -1, 2: 1})

    @property
    def real_dtype(self):
        return np.float32 if self.dtype == "f32" else np.float64

    @property
    def complex_dtype(self):
        return np.complex64 if self.dtype == "f32" else np.complex128

    def scaled(self, M: int | None = None, N: tuple | None = None,
               name: str | None = None) -> "Workload":
        """Same recipe with fewer points and/or modes."""
        return Workload(name or self.name, self.dim, tuple(N or self.N), int(M or self.M),
                        self.eps, self.dtype, self.types, self.dist, self.sigma,
                        self.seed, dict(self.iflag))


# The five benchmark workloads (sizes, tolerances, distributions).
WORKLOADS = {
    "2d_t1_f32_N64_M1e4": Workload("2d_t1_f32_N64_M1e4", 2, (64, 64), 10_000, 1e-5,
                                   "f32", (1,), "uniform", seed=0),
    "2d_f32_N1024_M1e7": Workload("2d_f32_N1024_M1e7", 2, (1024, 1024), 10_000_000, 1e-5,
                                  "f32", (1, 2), "uniform", seed=1),
    "2d_t1_f32_N1024_M1e7_cluster": Workload("2d_t1_f32_N1024_M1e7_cluster", 2, (1024, 1024),
                                             10_000_000, 1e-2, "f32", (1,), "cluster",
                                             sigma=0.05, seed=2),
    "3d_f32_N128_M3.2e7": Workload("3d_f32_N128_M3.2e7", 3, (128, 128, 128), 32_000_000,
                                   1e-6, "f32", (1, 2), "uniform", seed=3),
    "3d_f64_N64_M1e7_mix": Workload("3d_f64_N64_M1e7_mix", 3, (64, 64, 64), 10_000_000,
                                    1e-12, "f64", (1, 2), "mix", sigma=0.1, seed=4),
    # 1D (a "next" row): double precision at tolerance 1e-3 (w = 4), the
    # setting of the 1D sweeps in the finufft binsize discussion
    "1d_f64_N1e6_M1e7": Workload("1d_f64_N1e6_M1e7", 1, (1_000_000,), 10_000_000, 1e-3,
                                 "f64", (1, 2), "uniform", seed=5),
}


def _wrap(v: np.ndarray) -> np.ndarray:
    return np.mod(v + np.pi, TWO_PI) - np.pi


def sample(wl: Workload):
    """Points (x, y[, z]) and type 1 strengths c of the workload.

    One generator, seeded with ``wl.seed``, draws the coordinates in order x,
    y (, z) and then the real and imaginary parts of c."""
    rng = np.random.default_rng(wl.seed)
    M = wl.M
    if wl.dist == "uniform":
        pts = [rng.uniform(-np.pi, np.pi, M) for _ in range(wl.dim)]
    elif wl.dist == "cluster":
        pts = [_wrap(rng.normal(0.0, wl.sigma, M)) for _ in range(wl.dim)]
    elif wl.dist == "mix":
        h = M // 2
        pts = [np.concatenate([rng.uniform(-np.pi, np.pi, h),
                               _wrap(rng.normal(0.0, wl.sigma, M - h))])
               for _ in range(wl.dim)]
        order = rng.permutation(M)
        pts = [p[order] for p in pts]
    else:
        raise ValueError(f"unknown distribution {wl.dist!r}")
    re = rng.standard_normal(M)
    im = rng.standard_normal(M)
    c = (re + 1j * im).astype(wl.complex_dtype)
    return [p.astype(wl.real_dtype) for p in pts], c


def coefficients(wl: Workload) -> np.ndarray:
    """f_k for type 2: prod(N) complex values, k1 fastest (seed + 100)."""
    rng = np.random.default_rng(wl.seed + 100)
    K = int(np.prod(wl.N))
    re = rng.standard_normal(K)
    im = rng.standard_normal(K)
    return (re + 1j * im).astype(wl.complex_dtype)


def sha256(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()
