"""Scalar codebooks for one rotated coordinate (oracle; test infrastructure only).

After a random rotation of a unit vector in R^d, each coordinate is close to
N(0, 1/d) ([turbo4 post-mortem] section 5: "the 16-level optimal scalar quantizer
for the rotated-coordinate law N(0, 1/sqrt(d))", sigma = 1/sqrt(128) ~ 0.0884).
Two constructions are provided:

* QUANTILE: split the real line into 2^b cells of equal probability under
  N(0, sigma^2) and take each cell's conditional mean.  Section 5 of
  [turbo4 post-mortem] describes its d=128 table as "the conditional expectation
  within each quantile interval"; this construction reproduces the printed
  16-entry table to 4.4e-5.  In Lloyd terms it is one centroid step from the
  equal-probability partition, which is the reading under which "Lloyd
  iteration on N(0, 1/d)" reproduces that table.
* LLOYD: iterate Lloyd-Max (boundaries = midpoints, centroids = conditional
  means) from the QUANTILE start until it stops moving.
* SPHERE: the same Lloyd-Max iteration under the exact law of one coordinate of a
  uniformly random unit vector ("Lloyd-Max centroids for the rotated Beta
  distribution", [Triton deep dive] "write path and codebook"): density
  proportional to (1 - x^2)^((d-3)/2) on [-1, 1], i.e. (1 + x)/2 ~ Beta((d-1)/2,
  (d-1)/2).  Reading: the pages' "Beta(63.5, 63.5) for the absolute value" at
  d = 128 is this marginal written for (1 + x)/2 (the absolute value of a coordinate
  does not follow a symmetric Beta law).  At d=128, 16 levels
  its outer centroid is 2.733 sigma = 0.2416, the value quoted for the other
  implementation in section 9 of [turbo4 post-mortem]; for 1 and 2 bits the
  section-5 text says the reference uses the closed forms, which Lloyd reaches.

Readings (the pages are silent): turbo4 (16 levels) uses QUANTILE; turbo3
(8 levels) and the 2-bit MSE stage of the QJL "prod" keys use LLOYD.  Stored
tables are fp32 round-to-nearest of the fp64 centroids; decision boundaries are
the fp32 rounding of the fp64 midpoint of adjacent stored centroids.
"""

import math

import numpy as np

_SQRT2 = math.sqrt(2.0)


def _std_cdf(x):
    """Phi(x) for the standard normal, from erfc (libm)."""
    return 0.5 * math.erfc(-x / _SQRT2)


def _std_pdf(x):
    """phi(x) for the standard normal; 0 at +-inf."""
    if math.isinf(x):
        return 0.0
    return math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def _std_mass(a, b):
    """P(a < Z < b) for Z ~ N(0,1), evaluated on the side that avoids cancellation."""
    if a >= 0.0:
        return 0.5 * (math.erfc(a / _SQRT2) - math.erfc(b / _SQRT2))
    if b <= 0.0:
        return 0.5 * (math.erfc(-b / _SQRT2) - math.erfc(-a / _SQRT2))
    return 1.0 - 0.5 * math.erfc(-a / _SQRT2) - 0.5 * math.erfc(b / _SQRT2)


def std_normal_quantile(p):
    """Phi^{-1}(p) by bisection on erfc to an interval width below 1e-15."""
    if p <= 0.0:
        return -math.inf
    if p >= 1.0:
        return math.inf
    lo, hi = -40.0, 40.0
    while hi - lo > 1e-15:
        mid = 0.5 * (lo + hi)
        if mid == lo or mid == hi:
            break
        if _std_cdf(mid) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def _cond_mean_std(a, b):
    """E[Z | a < Z < b] for Z ~ N(0,1) = (phi(a) - phi(b)) / P(a < Z < b)."""
    return (_std_pdf(a) - _std_pdf(b)) / _std_mass(a, b)


def quantile_codebook(bits, d):
    """QUANTILE construction ([turbo4 post-mortem] section 5), fp64.

    Cells t_k = sigma * Phi^{-1}(k/K), k = 0..K, K = 2^bits, sigma = 1/sqrt(d);
    centroid c_k = E[X | t_k < X < t_{k+1}] for X ~ N(0, sigma^2).
    """
    K = 1 << bits
    sigma = 1.0 / math.sqrt(d)
    t = [std_normal_quantile(k / K) for k in range(K + 1)]
    return np.array([sigma * _cond_mean_std(t[k], t[k + 1]) for k in range(K)], dtype=np.float64)


def lloyd_codebook(bits, d, tol=1e-13, max_iter=1_000_000):
    """Converged Lloyd-Max quantizer for N(0, 1/d) ([turbo4 post-mortem] sections 5, 9), fp64.

    Starts from the QUANTILE centroids; each iteration sets the boundaries to the
    midpoints of adjacent centroids and the centroids to the conditional means of
    the resulting cells, until no centroid moves by more than ``tol``.
    """
    K = 1 << bits
    sigma = 1.0 / math.sqrt(d)
    c = quantile_codebook(bits, d) / sigma  # iterate in standard units
    for _ in range(max_iter):
        t = [-math.inf] + [0.5 * (c[k] + c[k + 1]) for k in range(K - 1)] + [math.inf]
        c_new = np.array([_cond_mean_std(t[k], t[k + 1]) for k in range(K)])
        moved = np.max(np.abs(c_new - c)) * sigma
        c = c_new
        if moved < tol:
            break
    return c * sigma


def _sphere_alpha(d):
    """Shape of the sphere marginal: (1 + X)/2 ~ Beta(alpha, alpha), alpha = (d - 1)/2."""
    return 0.5 * (d - 1)


def sphere_mass(a, b, d):
    """P(a < X < b) for one coordinate X of a uniform point on the unit sphere in R^d
    (density proportional to (1 - x^2)^((d - 3)/2) on [-1, 1]), through the regularized
    incomplete beta function of (1 + x)/2."""
    from scipy.special import betainc
    al = _sphere_alpha(d)
    ta = 0.0 if a <= -1.0 else (1.0 if a >= 1.0 else 0.5 * (1.0 + a))
    tb = 0.0 if b <= -1.0 else (1.0 if b >= 1.0 else 0.5 * (1.0 + b))
    if tb <= 0.5:  # both in the lower half: no cancellation against 1
        return float(betainc(al, al, tb) - betainc(al, al, ta))
    if ta >= 0.5:
        return float(betainc(al, al, 1.0 - ta) - betainc(al, al, 1.0 - tb))
    return float(1.0 - betainc(al, al, ta) - betainc(al, al, 1.0 - tb))


def sphere_cond_mean(a, b, d):
    """E[X | a < X < b] for the sphere marginal.  The first moment has a closed form,
    int x (1 - x^2)^m dx = -(1 - x^2)^(m+1) / (2 (m+1)), normalised by
    Z = int_{-1}^{1} (1 - x^2)^m dx = 2 4^m B(m+1, m+1), m = (d - 3)/2."""
    al = _sphere_alpha(d)  # = m + 1
    m = al - 1.0
    log_z = math.log(2.0) + m * math.log(4.0) + 2.0 * math.lgamma(al) - math.lgamma(2.0 * al)
    ga = (1.0 - a * a) ** al if -1.0 < a < 1.0 else 0.0
    gb = (1.0 - b * b) ** al if -1.0 < b < 1.0 else 0.0
    first = (ga - gb) / (2.0 * al) * math.exp(-log_z)
    return first / sphere_mass(a, b, d)


def sphere_codebook(bits, d, tol=1e-13, max_iter=1_000_000):
    """Converged Lloyd-Max quantizer for the exact law of a rotated unit-vector coordinate
    ([Triton deep dive] "write path and codebook": Lloyd-Max centroids for the rotated
    Beta distribution; (1 + x)/2 ~ Beta((d-1)/2, (d-1)/2) is the sphere marginal), fp64.

    Starts from the Gaussian QUANTILE centroids; boundaries = midpoints of adjacent
    centroids, centroids = conditional means of the cells under the sphere marginal,
    until no centroid moves by more than ``tol``.
    """
    K = 1 << bits
    c = quantile_codebook(bits, d)
    for _ in range(max_iter):
        t = [-1.0] + [0.5 * (c[k] + c[k + 1]) for k in range(K - 1)] + [1.0]
        c_new = np.array([sphere_cond_mean(t[k], t[k + 1], d) for k in range(K)])
        moved = np.max(np.abs(c_new - c))
        c = c_new
        if moved < tol:
            break
    return c


def make_codebook(bits, d, kind):
    """fp64 centroids of the requested kind ("quantile", "lloyd" or "sphere")."""
    if kind == "quantile":
        return quantile_codebook(bits, d)
    if kind == "lloyd":
        return lloyd_codebook(bits, d)
    if kind == "sphere":
        return sphere_codebook(bits, d)
    raise ValueError(f"unknown codebook kind {kind!r}")


def stored_codebook(centroids64):
    """Stored (fp32) centroids and decision boundaries.

    c32 = fp32 round-to-nearest of each fp64 centroid; b32[k] = fp32 rounding of
    the fp64 midpoint (c32[k] + c32[k+1]) / 2, k = 0..K-2.  Nearest-centroid
    encoding is idx = #{k : y > b32[k]} (strict), i.e. ties go to the lower index.
    """
    c32 = np.asarray(centroids64, dtype=np.float64).astype(np.float32)
    c64 = c32.astype(np.float64)
    b32 = ((c64[:-1] + c64[1:]) / 2.0).astype(np.float32)
    return c32, b32


def codebook_mse(centroids, d):
    """Exact mean-squared error E[(X - Q(X))^2] for X ~ N(0, 1/d) and nearest-centroid Q.

    Cells are bounded by the midpoints of adjacent centroids.  Per cell (a, b) in
    standard units, E[Z^2; cell] = P + a*phi(a) - b*phi(b), E[Z; cell] = phi(a) - phi(b).
    """
    sigma = 1.0 / math.sqrt(d)
    c = np.asarray(centroids, dtype=np.float64) / sigma
    K = len(c)
    t = [-math.inf] + [0.5 * (c[k] + c[k + 1]) for k in range(K - 1)] + [math.inf]
    total = 0.0
    for k in range(K):
        a, b = t[k], t[k + 1]
        mass = _std_mass(a, b)
        ez = _std_pdf(a) - _std_pdf(b)
        ez2 = mass + (0.0 if math.isinf(a) else a * _std_pdf(a)) - (0.0 if math.isinf(b) else b * _std_pdf(b))
        total += ez2 - 2.0 * c[k] * ez + c[k] * c[k] * mass
    return total * sigma * sigma
