"""Pins of the oracle's Lloyd-Max codebook (CPU only).

The pages print no codebook values, so the pins are what the mathematics
fixes: closed forms at d = 3 and b = 1, the Lloyd-Max fixed-point conditions
re-checked with independent numerical quadrature, symmetry, the second moment
1/d of the density, monotone distortion, and the Gaussian high-dimension
limit recomputed here from the normal law.
"""
import math

import numpy as np
import pytest
from scipy import integrate, stats

import oracle


def _pdf(d):
    cd = math.exp(math.lgamma(d / 2) - 0.5 * math.log(math.pi) - math.lgamma((d - 1) / 2))
    return lambda x: cd * (1 - x * x) ** ((d - 3) / 2)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6])
def test_d3_density_is_uniform_so_codebook_is_uniform(bits):
    cb = oracle.lloyd_max(3, bits)
    k = 1 << bits
    expect = -1 + (2 * np.arange(k) + 1) / k
    np.testing.assert_allclose(cb.centroids, expect, atol=1e-13)
    # uniform quantizer of step 2/k on a unit-density-1/2 interval: MSE = step^2/12
    assert cb.mse_per_coord == pytest.approx((2 / k) ** 2 / 12, rel=1e-10)


@pytest.mark.parametrize("d", [4, 16, 64, 128, 256])
def test_one_bit_closed_form(d):
    cb = oracle.lloyd_max(d, 1)
    e_abs = math.exp(math.lgamma(d / 2) - 0.5 * math.log(math.pi) - math.lgamma((d + 1) / 2))
    np.testing.assert_allclose(cb.centroids, [-e_abs, e_abs], rtol=1e-13)
    assert cb.thresholds[0] == 0.0
    assert cb.mse_per_coord == pytest.approx(1 / d - e_abs ** 2, rel=1e-11)


@pytest.mark.parametrize("d,bits", [(16, 2), (64, 3), (128, 2), (128, 3), (128, 4), (256, 4)])
def test_lloyd_max_fixed_point_by_quadrature(d, bits):
    cb = oracle.lloyd_max(d, bits)
    f = _pdf(d)
    c, t = cb.centroids, cb.thresholds
    np.testing.assert_allclose(t, (c[:-1] + c[1:]) / 2, rtol=0, atol=1e-17)
    edges = np.concatenate([[-1.0], t, [1.0]])
    for k in range(len(c)):
        m0 = integrate.quad(f, edges[k], edges[k + 1], epsabs=1e-15, epsrel=1e-14, limit=200)[0]
        m1 = integrate.quad(lambda x: x * f(x), edges[k], edges[k + 1], epsabs=1e-16, epsrel=1e-14, limit=200)[0]
        assert abs(m1 / m0 - c[k]) < 1e-12, (k, m1 / m0, c[k])


@pytest.mark.parametrize("d,bits", [(8, 3), (128, 3), (128, 4)])
def test_symmetric_and_sorted(d, bits):
    cb = oracle.lloyd_max(d, bits)
    c = cb.centroids
    np.testing.assert_array_equal(c, -c[::-1])
    assert np.all(np.diff(c) > 0)
    assert np.all(np.diff(cb.thresholds) > 0)
    np.testing.assert_array_equal(cb.centroids32, c.astype(np.float32))


@pytest.mark.parametrize("d", [8, 32, 128])
def test_second_moment_of_density_is_one_over_d(d):
    f = _pdf(d)
    total = integrate.quad(f, -1, 1, epsrel=1e-13, limit=200)[0]
    m2 = integrate.quad(lambda x: x * x * f(x), -1, 1, epsrel=1e-13, limit=200)[0]
    assert total == pytest.approx(1.0, rel=1e-9)
    assert m2 == pytest.approx(1.0 / d, rel=1e-9)


@pytest.mark.parametrize("d", [16, 128])
def test_mse_matches_quadrature_and_falls_with_bits(d):
    f = _pdf(d)
    prev = math.inf
    for bits in range(1, 6):
        cb = oracle.lloyd_max(d, bits)
        edges = np.concatenate([[-1.0], cb.thresholds, [1.0]])
        mse = sum(integrate.quad(lambda x, ck=ck: (x - ck) ** 2 * f(x), edges[k], edges[k + 1],
                                 epsabs=1e-17, epsrel=1e-13, limit=200)[0]
                  for k, ck in enumerate(cb.centroids))
        assert cb.mse_per_coord == pytest.approx(mse, rel=1e-9)
        assert cb.mse_per_coord < prev
        prev = cb.mse_per_coord


def _gaussian_lloyd_max_distortion(bits, iters=20000):
    k = 1 << bits
    c = stats.norm.ppf((np.arange(k) + 0.5) / k)
    for _ in range(iters):
        t = (c[:-1] + c[1:]) / 2
        e = np.concatenate([[-np.inf], t, [np.inf]])
        mass = stats.norm.cdf(e[1:]) - stats.norm.cdf(e[:-1])
        c_new = (stats.norm.pdf(e[:-1]) - stats.norm.pdf(e[1:])) / mass
        if np.max(np.abs(c_new - c)) < 1e-14:
            c = c_new
            break
        c = c_new
    t = (c[:-1] + c[1:]) / 2
    e = np.concatenate([[-np.inf], t, [np.inf]])
    pe = np.where(np.isfinite(e), stats.norm.pdf(e), 0.0)
    ee = np.where(np.isfinite(e), e, 0.0)
    m0 = stats.norm.cdf(e[1:]) - stats.norm.cdf(e[:-1])
    m1 = pe[:-1] - pe[1:]
    m2 = m0 + ee[:-1] * pe[:-1] - ee[1:] * pe[1:]
    return float(np.sum(m2 - 2 * c * m1 + c * c * m0))


def test_one_bit_gaussian_distortion_closed_form():
    assert _gaussian_lloyd_max_distortion(1) == pytest.approx(1 - 2 / math.pi, rel=1e-12)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_high_dimension_limit_is_gaussian_lloyd_max(bits):
    g = _gaussian_lloyd_max_distortion(bits)
    d = 4096
    assert d * oracle.lloyd_max(d, bits).mse_per_coord == pytest.approx(g, rel=2e-3)
    # and the approach is monotone in d
    gaps = [abs(dd * oracle.lloyd_max(dd, bits).mse_per_coord - g) for dd in (64, 256, 1024)]
    assert gaps[0] > gaps[1] > gaps[2]


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_threshold_rule_is_nearest_centroid(bits):
    cb = oracle.lloyd_max(128, bits)
    y = np.random.default_rng(bits).standard_normal(200000).astype(np.float32) / np.float32(math.sqrt(128))
    rule = (y[:, None] >= cb.thresholds32[None, :]).sum(axis=1)
    brute = np.argmin(np.abs(y.astype(np.float64)[:, None] - cb.centroids32.astype(np.float64)[None, :]), axis=1)
    differ = rule != brute
    # only where y sits between the exact float32 midpoint and its rounding
    if differ.any():
        gap = np.min(np.abs(y[differ, None].astype(np.float64) - cb.thresholds[None, :]), axis=1)
        assert np.all(gap < 1e-7)
    assert differ.mean() < 1e-5
