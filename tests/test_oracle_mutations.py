"""The oracle's pins are sharp enough: plausible mistakes planted in the oracle
(on the CPU, by monkeypatching one step) make at least one pin fail.

Each mutation corrupts one step of the three-step scheme of "cuFINUFFT: a
load-balanced GPU library for general-purpose nonuniform FFTs" (Sec. II); the
checks are the closed forms and the accuracy claim used in test_oracle_pins.
"""
import numpy as np
import pytest

import oracle


def _single_point_ok(eps=1e-9, N=(12, 8)):
    x0 = [0.7, -2.1]
    f = oracle.nufft_type1([[v] for v in x0], [1.0], N, eps, -1)
    ks = np.meshgrid(*[np.arange(-(n // 2), n - n // 2) for n in reversed(N)], indexing="ij")
    ref = np.exp(-1j * sum(k * v for k, v in zip(reversed(ks), x0)))
    return oracle.rel_l2(f, ref) < 20 * eps


def _sweep_ok(eps=1e-6, N=(20, 16), M=500):
    rng = np.random.default_rng(1)
    pts = [rng.uniform(-np.pi, np.pi, M) for _ in N]
    c = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    e = oracle.rel_l2(oracle.nufft_type1(pts, c, N, eps, -1), oracle.direct_type1(pts, c, N, -1))
    return eps / 4 <= e <= 4 * eps


def _adjoint_ok(N=(10, 6)):
    rng = np.random.default_rng(2)
    pts = [rng.uniform(-np.pi, np.pi, 50) for _ in N]
    c = rng.standard_normal(50) + 1j * rng.standard_normal(50)
    f = rng.standard_normal(60) + 1j * rng.standard_normal(60)
    lhs = np.vdot(oracle.nufft_type1(pts, c, N, 1e-6, 1).ravel(), f)
    rhs = np.vdot(c, oracle.nufft_type2(pts, f, N, 1e-6, -1))
    return abs(lhs - rhs) <= 1e-12 * abs(lhs)


def _all_pins_ok():
    return _single_point_ok() and _sweep_ok() and _adjoint_ok()


def test_unmutated_oracle_passes():
    assert _all_pins_ok()


def _mut_fft_sign(monkeypatch):
    orig = oracle._fft
    monkeypatch.setattr(oracle, "_fft", lambda b, iflag: orig(b, -iflag))


def _mut_no_correction(monkeypatch):
    monkeypatch.setattr(oracle, "correction_factors",
                        lambda N, n, w, beta: np.ones(N))


def _mut_correction_inverted(monkeypatch):
    orig = oracle.correction_factors
    monkeypatch.setattr(oracle, "correction_factors",
                        lambda N, n, w, beta: 1.0 / orig(N, n, w, beta))


def _mut_width_minus_one(monkeypatch):
    orig = oracle.es_params
    monkeypatch.setattr(oracle, "es_params",
                        lambda eps, sigma=2.0: (orig(eps)[0] - 1, 2.30 * (orig(eps)[0] - 1)))


def _mut_transposed_modes(monkeypatch):
    orig = oracle._fine_index
    # read the fine grid at -k instead of k
    monkeypatch.setattr(oracle, "_fine_index", lambda N, n: orig(N, n)[::-1] % n)


def _mut_mode_offset(monkeypatch):
    orig = oracle.mode_indices
    monkeypatch.setattr(oracle, "mode_indices", lambda N: orig(N) + 1)


def _mut_phihat_scaled(monkeypatch):
    orig = oracle.phihat
    monkeypatch.setattr(oracle, "phihat", lambda xi, beta, q=200: orig(np.asarray(xi) * 1.05, beta, q))


def _sigma_sweep_ok(eps=1e-6, N=(48, 40), M=1500, sigma=1.25):
    rng = np.random.default_rng(3)
    pts = [rng.uniform(-np.pi, np.pi, M) for _ in N]
    c = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    e = oracle.rel_l2(oracle.nufft_type1(pts, c, N, eps, -1, sigma),
                      oracle.direct_type1(pts, c, N, -1))
    return eps / 8 <= e <= 3 * eps


def _mut_sigma_beta_of_two(monkeypatch):
    orig = oracle.es_params
    # the sigma < 2 width with the sigma = 2 shape beta = 2.30 w
    monkeypatch.setattr(oracle, "es_params",
                        lambda eps, sigma=2.0: (orig(eps, sigma)[0], 2.30 * orig(eps, sigma)[0]))


def _mut_sigma_grid_of_two(monkeypatch):
    orig = oracle.fine_grid_size
    # the sigma < 2 kernel on the sigma = 2 grid
    monkeypatch.setattr(oracle, "fine_grid_size", lambda N, w, sigma=2.0: orig(N, w))


def _mut_sigma_width_of_two(monkeypatch):
    orig = oracle.es_params
    # eq. (6) width for every sigma, with the sigma < 2 beta scaling
    monkeypatch.setattr(oracle, "es_params",
                        lambda eps, sigma=2.0: (orig(eps)[0],
                                                orig(eps, sigma)[1] / orig(eps, sigma)[0] * orig(eps)[0]))


@pytest.mark.parametrize("mutate", [_mut_sigma_beta_of_two, _mut_sigma_grid_of_two,
                                    _mut_sigma_width_of_two])
def test_planted_sigma_mistake_is_caught(monkeypatch, mutate):
    assert _sigma_sweep_ok()
    mutate(monkeypatch)
    assert not _sigma_sweep_ok()


@pytest.mark.parametrize("mutate", [_mut_fft_sign, _mut_no_correction, _mut_correction_inverted,
                                    _mut_width_minus_one, _mut_transposed_modes, _mut_mode_offset,
                                    _mut_phihat_scaled])
def test_planted_mistake_is_caught(monkeypatch, mutate):
    mutate(monkeypatch)
    assert not _all_pins_ok()
