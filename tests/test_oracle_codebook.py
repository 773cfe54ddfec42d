"""Pins of the oracle's codebooks against printed values, textbook tables and integrals."""

import math

import numpy as np
import pytest
from scipy import integrate, stats

import oracle
from conftest import golden_lines

D = 128
SIGMA = 1.0 / math.sqrt(D)


def printed_table():
    return np.array([float(v) for v in golden_lines("turbo4_centroids_d128.txt")])


def max_table():
    rows = {}
    for ln in golden_lines("max_gaussian_quantizer.txt"):
        parts = ln.split()
        K = int(parts[0])
        rows[K] = (float(parts[1]), np.array([float(v) for v in parts[2:]]))
    return rows


def test_quantile_reproduces_printed_turbo4_table():
    """One Lloyd step from equal-probability cells gives the printed d=128 table.

    The table has 4 decimals, so every entry must agree to the rounding half-unit
    5e-5 (spec bound 1e-3)."""
    c = oracle.quantile_codebook(4, D)
    assert np.max(np.abs(c - printed_table())) <= 5.0e-5 + 1e-9


def test_printed_sigma_and_outer_centroid(page_numbers):
    assert abs(SIGMA - page_numbers["sigma_d128"]) < 5e-5
    c = oracle.quantile_codebook(4, D)
    assert abs(c[-1] / SIGMA - page_numbers["table_outer_in_sigma"]) < 5e-3


@pytest.mark.parametrize("kind", ["quantile", "lloyd"])
def test_one_bit_closed_form(kind):
    """1-bit codebook = +-sqrt(2/(pi d)) (the paper's closed form)."""
    c = oracle.make_codebook(1, D, kind)
    ref = math.sqrt(2.0 / (math.pi * D))
    assert np.allclose(c, [-ref, ref], rtol=0, atol=1e-12)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_lloyd_matches_max_gaussian_quantizer(bits):
    """Converged Lloyd on N(0, 1/d), rescaled to unit variance, is Max's 1960 quantizer."""
    K = 1 << bits
    dist, levels = max_table()[K]
    c = oracle.lloyd_codebook(bits, D) / SIGMA
    assert np.allclose(c[K // 2:], levels, rtol=0, atol=6e-4)
    mse = oracle.codebook_mse(oracle.lloyd_codebook(bits, D), D) * D
    assert abs(mse - dist) / dist < 1e-3


def test_lloyd16_outer_matches_other_implementation(page_numbers):
    """Section 9: the converged Gaussian 16-level outer centroid is 0.2416 = 2.73 sigma."""
    c = oracle.lloyd_codebook(4, D)
    assert abs(c[-1] - page_numbers["lloyd16_outer_d128"]) < 1e-4
    assert abs(c[-1] / SIGMA - page_numbers["lloyd16_outer_in_sigma"]) < 5e-3


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_lloyd_is_fixed_point_by_quadrature(bits):
    """Each converged centroid is the conditional mean of its midpoint cell (scipy quad)."""
    c = oracle.lloyd_codebook(bits, D)
    t = [-np.inf] + list((c[:-1] + c[1:]) / 2) + [np.inf]
    pdf = stats.norm(0.0, SIGMA).pdf
    for k in range(len(c)):
        mass = integrate.quad(pdf, t[k], t[k + 1], epsabs=1e-14, epsrel=1e-13)[0]
        mom = integrate.quad(lambda x: x * pdf(x), t[k], t[k + 1], epsabs=1e-14, epsrel=1e-13)[0]
        assert abs(mom / mass - c[k]) < 1e-10


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_quantile_cells_have_equal_mass_by_quadrature(bits):
    """QUANTILE: each centroid is the conditional mean of an equal-probability cell."""
    K = 1 << bits
    c = oracle.quantile_codebook(bits, D)
    t = [stats.norm.ppf(k / K, scale=SIGMA) for k in range(K + 1)]
    pdf = stats.norm(0.0, SIGMA).pdf
    for k in range(K):
        mom = integrate.quad(lambda x: x * pdf(x), t[k], t[k + 1], epsabs=1e-14, epsrel=1e-13)[0]
        assert abs(mom * K - c[k]) < 1e-10


@pytest.mark.parametrize("kind", ["quantile", "lloyd", "sphere"])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_symmetric_and_increasing(kind, bits):
    c = oracle.make_codebook(bits, D, kind)
    assert np.all(np.diff(c) > 0)
    assert np.allclose(c, -c[::-1], atol=1e-15)


def test_mse_quantile_vs_lloyd_and_monte_carlo():
    """Per-coordinate MSE x d: QUANTILE-16 ~ 0.0203, LLOYD-16 ~ 0.0095 (exact and Monte Carlo)."""
    q = oracle.quantile_codebook(4, D)
    l = oracle.lloyd_codebook(4, D)
    mq = oracle.codebook_mse(q, D) * D
    ml = oracle.codebook_mse(l, D) * D
    assert abs(mq - 0.0203) < 5e-4
    assert abs(ml - 0.0095) < 5e-5
    rng = np.random.default_rng(11)
    y = rng.normal(0.0, SIGMA, size=2_000_000)
    for c, exact in ((q, mq), (l, ml)):
        c32, b32 = oracle.stored_codebook(c)
        idx = (y[:, None] > b32.astype(np.float64)).sum(1)
        mc = np.mean((y - c32[idx]) ** 2) * D
        assert abs(mc - exact) / exact < 0.01


@pytest.mark.parametrize("kind", ["quantile", "lloyd"])
def test_stored_boundaries_are_midpoints_and_encode_is_nearest(kind):
    """Boundaries are the midpoints rounded to fp32; counting boundaries is nearest-centroid."""
    from oracle.formats import nearest_index
    c32, b32 = oracle.stored_codebook(oracle.make_codebook(4, D, kind))
    assert c32.dtype == np.float32 and b32.dtype == np.float32
    c64 = c32.astype(np.float64)
    mid = (c64[:-1] + c64[1:]) / 2
    ulp = np.spacing(np.abs(b32)).astype(np.float64)
    assert np.all(np.abs(b32.astype(np.float64) - mid) <= ulp / 2)
    rng = np.random.default_rng(5)
    y = np.concatenate([rng.normal(0, 2 * SIGMA, 200_000), c64])
    idx = nearest_index(y, b32)
    brute = np.argmin(np.abs(y[:, None] - c64[None, :]), axis=1)
    assert np.array_equal(idx, brute)
    # a coordinate exactly on a boundary goes to the lower index
    assert np.array_equal(nearest_index(b32.astype(np.float64), b32), np.arange(15))
    assert np.array_equal(nearest_index(b32, b32), np.arange(15))


# ---- sphere-marginal (rotated unit-vector coordinate) codebook

def _sphere_pdf(d):
    m = 0.5 * (d - 3)
    z = integrate.quad(lambda x: (1 - x * x) ** m, -1, 1, epsabs=0, epsrel=1e-13)[0]
    return lambda x: (1 - x * x) ** m / z


def test_sphere_one_bit_closed_form():
    """1 bit: the centroid of x > 0 is E|X| = Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2))."""
    for d in (8, 128, 1024):
        c = oracle.sphere_codebook(1, d)
        exact = math.exp(math.lgamma(d / 2) - math.lgamma((d + 1) / 2)) / math.sqrt(math.pi)
        assert abs(c[1] - exact) < 1e-12 and abs(c[0] + exact) < 1e-12


def test_sphere_law_mass_and_variance():
    """The marginal has unit mass and variance exactly 1/d (E X^2 = 1/d on the sphere)."""
    assert abs(oracle.sphere_mass(-1.0, 1.0, D) - 1.0) < 1e-14
    f = _sphere_pdf(D)
    var = integrate.quad(lambda x: x * x * f(x), -1, 1, epsabs=0, epsrel=1e-12)[0]
    assert abs(var - 1.0 / D) < 1e-13
    for a, b in ((-0.3, -0.1), (-0.05, 0.02), (0.1, 0.45)):
        q = integrate.quad(f, a, b, epsabs=0, epsrel=1e-13)[0]
        assert abs(oracle.sphere_mass(a, b, D) - q) < 1e-13


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_sphere_lloyd_is_fixed_point_by_quadrature(bits):
    """Each centroid is the conditional mean of its midpoint cell, by direct quadrature of
    the density (independent of the incomplete-beta route the codebook takes)."""
    c = oracle.sphere_codebook(bits, D)
    f = _sphere_pdf(D)
    t = [-1.0] + list((c[:-1] + c[1:]) / 2) + [1.0]
    for k in range(len(c)):
        mass = integrate.quad(f, t[k], t[k + 1], epsabs=0, epsrel=1e-13)[0]
        mom = integrate.quad(lambda x: x * f(x), t[k], t[k + 1], epsabs=0, epsrel=1e-13)[0]
        assert abs(mom / mass - c[k]) < 1e-10


def test_sphere_codebook_tends_to_gaussian_lloyd():
    """The sphere marginal tends to N(0, 1/d): scaled by sqrt(d) the two codebooks meet as
    d grows (and differ at d = 128 by the 4th decimal)."""
    for bits in (2, 4):
        gap = [np.max(np.abs(oracle.sphere_codebook(bits, d) - oracle.lloyd_codebook(bits, d))) * math.sqrt(d)
               for d in (128, 16384)]
        assert gap[1] < gap[0] / 50 and gap[1] < 1e-3


def test_sphere_codebook_beats_gaussian_lloyd_on_the_sphere_law():
    """Lloyd-Max optimality: under the sphere marginal, the sphere codebook's distortion is
    below the Gaussian codebook's (quadrature of both)."""
    f = _sphere_pdf(D)

    def mse(c):
        t = [-1.0] + list((c[:-1] + c[1:]) / 2) + [1.0]
        return sum(integrate.quad(lambda x: (x - c[k]) ** 2 * f(x), t[k], t[k + 1], epsabs=0, epsrel=1e-12)[0]
                   for k in range(len(c)))
    for bits in (3, 4):
        assert mse(oracle.sphere_codebook(bits, D)) < mse(oracle.lloyd_codebook(bits, D))
