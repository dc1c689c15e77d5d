"""Pins of the calibration oracle (``oracle/calibration.py``) against exact
rational arithmetic, closed forms, planted spectra, order-statistic brute force
and a Gaussian quantile from the library's normal distribution.  Each pin takes
the oracle module, so a planted-mistake copy can be run through the same pins.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def bf16_bits(x) -> np.ndarray:
    """fp64 values that are exact in bf16 -> bit patterns (asserts exactness)."""
    f = np.asarray(x, dtype=np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, f), "value not exact in bf16"
    return bits


def bf16_round_bits(x) -> np.ndarray:
    """Round fp64 values to bf16 (nearest even via fp32) -> bit patterns."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def haar(D: int, rng: np.random.Generator) -> np.ndarray:
    q, r = np.linalg.qr(rng.standard_normal((D, D)))
    return q * np.sign(np.diag(r))


def sign_rule(R: np.ndarray) -> np.ndarray:
    """Flip each column so that its first largest-magnitude entry is positive."""
    R = R.copy()
    for j in range(R.shape[1]):
        i = int(np.argmax(np.abs(R[:, j])))
        if R[i, j] < 0:
            R[:, j] = -R[:, j]
    return R


# ---- (C1) covariance -------------------------------------------------------------

def pin_covariance_closed_form(cal):
    # samples (1, 2) and (3, 4): second moment [[5, 7], [7, 10]], covariance all ones
    x = bf16_bits(np.array([[[1.0, 2.0]], [[3.0, 4.0]]]))
    np.testing.assert_array_equal(cal.covariance(x, centered=False)[0], [[5.0, 7.0], [7.0, 10.0]])
    np.testing.assert_array_equal(cal.covariance(x, centered=True)[0], [[1.0, 1.0], [1.0, 1.0]])


def pin_covariance_exact_rationals(cal):
    rng = np.random.default_rng(5)
    N, H, D = 7, 2, 5
    ints = rng.integers(-9, 10, size=(N, H, D))
    x = bf16_bits(ints.astype(np.float64))
    for centered in (False, True):
        got = cal.covariance(x, centered)
        for h in range(H):
            mu = [Fraction(int(sum(ints[t, h, i] for t in range(N))), N) for i in range(D)]
            for i in range(D):
                for j in range(D):
                    acc = Fraction(0)
                    for t in range(N):
                        a = Fraction(int(ints[t, h, i])) - (mu[i] if centered else 0)
                        b = Fraction(int(ints[t, h, j])) - (mu[j] if centered else 0)
                        acc += a * b
                    exact = acc / N
                    assert abs(got[h, i, j] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact))), \
                        (centered, h, i, j, got[h, i, j], exact)


def pin_covariance_shift_invariance(cal):
    # adding one vector to every sample leaves the covariance unchanged (exact in bf16: small ints)
    rng = np.random.default_rng(6)
    ints = rng.integers(-8, 9, size=(12, 1, 4)).astype(np.float64)
    shift = np.array([3.0, -5.0, 7.0, 1.0])
    a = cal.covariance(bf16_bits(ints), centered=True)
    b = cal.covariance(bf16_bits(ints + shift), centered=True)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    # and the second moment changes by exactly the outer-product terms
    m0 = cal.covariance(bf16_bits(ints), centered=False)[0]
    m1 = cal.covariance(bf16_bits(ints + shift), centered=False)[0]
    mu = ints[:, 0, :].mean(axis=0)
    expect = m0 + np.outer(mu, shift) + np.outer(shift, mu) + np.outer(shift, shift)
    np.testing.assert_allclose(m1, expect, rtol=0, atol=1e-12)


# ---- (C2) rotation ---------------------------------------------------------------

def pin_rotation_diagonal_is_sorting_permutation(cal):
    C = np.diag([3.0, 1.0, 4.0, 2.0])[None]
    R, lam = cal.rotation(C)
    np.testing.assert_array_equal(lam[0], [4.0, 3.0, 2.0, 1.0])
    P = np.zeros((4, 4))
    for col, src in enumerate([2, 0, 3, 1]):
        P[src, col] = 1.0
    np.testing.assert_array_equal(R[0], P)


def pin_rotation_2x2_closed_form(cal):
    a, b = 5.0, 2.0
    R, lam = cal.rotation(np.array([[[a, b], [b, a]]]))
    np.testing.assert_allclose(lam[0], [a + b, a - b], rtol=0, atol=1e-14)
    r = 1.0 / math.sqrt(2.0)
    # eigenvector of a + b is (1, 1); of a - b is (1, -1) (tie in magnitude: the lower row is positive)
    np.testing.assert_allclose(R[0], [[r, r], [r, -r]], rtol=0, atol=1e-14)


def pin_rotation_planted_spectrum(cal):
    rng = np.random.default_rng(7)
    H, D = 2, 16
    C = np.zeros((H, D, D))
    Q = np.zeros((H, D, D))
    lam_true = np.zeros((H, D))
    for h in range(H):
        lam_true[h] = np.sort(rng.uniform(1.0, 50.0, D))[::-1] + np.arange(D)[::-1] * 0.5
        Q[h] = sign_rule(haar(D, rng))
        C[h] = Q[h] @ np.diag(lam_true[h]) @ Q[h].T
    R, lam = cal.rotation(C)
    np.testing.assert_allclose(lam, lam_true, rtol=1e-12, atol=0)
    np.testing.assert_allclose(R, Q, rtol=0, atol=1e-10)


def pin_rotation_invariants(cal):
    rng = np.random.default_rng(8)
    x = bf16_round_bits(rng.standard_normal((300, 3, 8)) * np.linspace(0.5, 4.0, 8))
    C = cal.covariance(x, True)
    R, lam = cal.rotation(C)
    for h in range(3):
        np.testing.assert_allclose(R[h].T @ R[h], np.eye(8), rtol=0, atol=1e-12)
        np.testing.assert_allclose(R[h].T @ C[h] @ R[h], np.diag(lam[h]), rtol=0, atol=1e-12 * lam[h, 0])
        assert np.all(np.diff(lam[h]) <= 0), "eigenvalues not descending"
        for j in range(8):
            i = int(np.argmax(np.abs(R[h][:, j])))
            assert R[h][i, j] > 0, "sign rule"
        # spectral identities: trace, Frobenius norm and determinant
        assert abs(np.sum(lam[h]) - np.trace(C[h])) <= 1e-12 * lam[h, 0] * 8
        assert abs(np.sum(lam[h] ** 2) - np.sum(C[h] ** 2)) <= 1e-12 * lam[h, 0] ** 2 * 8
        assert abs(np.prod(lam[h]) / np.linalg.det(C[h]) - 1.0) <= 1e-9


def pin_rotation_decorrelates_samples(cal):
    # the rotated calibration samples have a diagonal covariance with the eigenvalues on it
    rng = np.random.default_rng(9)
    A = rng.standard_normal((6, 6))
    x = bf16_round_bits(rng.standard_normal((500, 1, 6)) @ A + np.array([1.0, -2.0, 0.5, 3.0, 0.0, 1.5]))
    C = cal.covariance(x, True)
    R, lam = cal.rotation(C)
    y = cal.bf16_bits_to_f64(x)[:, 0, :] @ R[0]
    yc = y - y.mean(axis=0)
    np.testing.assert_allclose(yc.T @ yc / y.shape[0], np.diag(lam[0]), rtol=0, atol=1e-10 * lam[0, 0])


# ---- (C3) clipping thresholds -----------------------------------------------------

def _brute_kth(values, k):
    """k-th smallest (1-based) by counting: the v with #{< v} < k <= #{<= v}."""
    vals = list(values)
    for v in vals:
        below = sum(1 for u in vals if u < v)
        at_most = sum(1 for u in vals if u <= v)
        if below < k <= at_most:
            return v
    raise AssertionError("no order statistic")


def pin_quantile_index(cal):
    assert cal.quantile_index(1.0, 10) == 10
    assert cal.quantile_index(0.5, 10) == 5
    assert cal.quantile_index(0.51, 10) == 6
    assert cal.quantile_index(1e-9, 10) == 1
    assert cal.quantile_index(0.999, 1000) == 999
    assert cal.quantile_index(0.9995, 1000) == 1000


def pin_clip_brute_force(cal):
    rng = np.random.default_rng(10)
    N, H, D = 11, 2, 4
    x = bf16_round_bits(rng.standard_normal((N, H, D)) * 3.0)
    R = np.stack([haar(D, rng) for _ in range(H)])
    xv = cal.bf16_bits_to_f64(x)
    for q in (1.0, 0.5, 0.7, 1.0 / N):
        got = cal.clip_thresholds(x, R, q)
        k = math.ceil(q * N)
        for h in range(H):
            for j in range(D):
                mags = [abs(sum(xv[t, h, i] * R[h, i, j] for i in range(D))) for t in range(N)]
                assert abs(got[h, j] - _brute_kth(mags, k)) <= 1e-12 * max(mags), (q, h, j)


def pin_clip_identity_extremes(cal):
    # R = I: q = 1 gives max |x_j|, q = 1/N gives min |x_j| (hand-checked small integers)
    x = bf16_bits(np.array([[[-4.0, 1.0]], [[2.0, -3.0]], [[1.0, 0.5]]]))
    I = np.eye(2)[None]
    np.testing.assert_array_equal(cal.clip_thresholds(x, I, 1.0)[0], [4.0, 3.0])
    np.testing.assert_array_equal(cal.clip_thresholds(x, I, 1.0 / 3.0)[0], [1.0, 0.5])
    np.testing.assert_array_equal(cal.clip_thresholds(x, I, 0.5)[0], [2.0, 1.0])


def pin_calibrate_gaussian_quantiles(cal):
    # samples ~ N(0, Q diag(lam) Q^T): the rotated channel j is N(0, lam_j), so its
    # q-quantile of |y| approaches sqrt(lam_j) * Phi^-1((1 + q) / 2)
    from scipy.stats import norm
    rng = np.random.default_rng(11)
    D, N = 8, 40000
    lam = np.array([64.0, 36.0, 16.0, 9.0, 4.0, 2.0, 1.0, 0.25])
    Q = haar(D, rng)
    z = rng.standard_normal((N, D)) * np.sqrt(lam)
    x = bf16_round_bits((z @ Q.T)[:, None, :])
    q = 0.9
    C, R, lam_hat, clip = cal.calibrate(x, centered=True, q=q)
    np.testing.assert_allclose(lam_hat[0], lam, rtol=0.05)
    np.testing.assert_allclose(clip[0], np.sqrt(lam) * norm.ppf((1 + q) / 2), rtol=0.04)
    # the principal directions are recovered (the spectrum is well separated)
    overlap = np.abs(np.sum(R[0] * Q, axis=0))
    assert np.all(overlap[:5] > 0.99), overlap


def pin_calibrate_uses_given_rotation_columns(cal):
    # a planted anisotropic rotation: clip from R's columns (not rows) separates the channels
    rng = np.random.default_rng(12)
    D, N = 4, 4000
    lam = np.array([100.0, 25.0, 4.0, 1.0])
    Q = sign_rule(haar(D, rng))
    x = bf16_round_bits(((rng.standard_normal((N, D)) * np.sqrt(lam)) @ Q.T)[:, None, :])
    clip = cal.clip_thresholds(x, Q[None], 1.0)[0]
    xv = cal.bf16_bits_to_f64(x)[:, 0, :]
    for j in range(D):
        assert abs(clip[j] - np.max(np.abs(xv @ Q[:, j]))) <= 1e-12 * clip[j]
    assert clip[0] > 3 * clip[2]


ALL_PINS = [
    pin_covariance_closed_form,
    pin_covariance_exact_rationals,
    pin_covariance_shift_invariance,
    pin_rotation_diagonal_is_sorting_permutation,
    pin_rotation_2x2_closed_form,
    pin_rotation_planted_spectrum,
    pin_rotation_invariants,
    pin_rotation_decorrelates_samples,
    pin_quantile_index,
    pin_clip_brute_force,
    pin_clip_identity_extremes,
    pin_calibrate_gaussian_quantiles,
    pin_calibrate_uses_given_rotation_columns,
]
