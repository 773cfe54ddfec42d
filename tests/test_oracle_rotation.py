"""Pins of the oracle's rotations, generator and QJL matrix."""

import math

import numpy as np
import pytest
from scipy import linalg, stats

import oracle
from conftest import golden_lines
from oracle.formats import Rotation

D = 128


def test_splitmix64_known_answers():
    ref = [int(v, 16) for v in golden_lines("splitmix64_seed0.txt")]
    out = [int(v) for v in oracle.splitmix64(0, len(ref))]
    assert out == ref


def test_splitmix64_is_counter_based():
    full = oracle.splitmix64(1234, 40)
    assert np.array_equal(oracle.splitmix64(1234, 10, start=30), full[30:])


def test_fwht_is_sylvester_hadamard():
    """FWHT(e_j) is column j of the Sylvester Hadamard matrix (scipy.linalg.hadamard)."""
    H = linalg.hadamard(D).astype(np.float64)
    assert np.array_equal(oracle.fwht(np.eye(D)), H.T)  # row j of the result is H e_j
    assert np.array_equal(H @ H.T, D * np.eye(D))
    x = np.random.default_rng(0).standard_normal((7, D))
    assert np.allclose(oracle.fwht(x), x @ H.T, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 5, 2**63 + 7])
def test_randomized_wht_orthogonal_and_fp32_close(seed):
    s = oracle.wht_signs(seed, D)
    assert set(np.unique(s)) <= {-1.0, 1.0}
    R = oracle.wht_rotation_matrix(s)
    assert np.max(np.abs(R.T @ R - np.eye(D))) < 1e-12
    H = linalg.hadamard(D).astype(np.float64)
    assert np.allclose(R, H @ np.diag(s) / math.sqrt(D), atol=1e-15)
    u = np.random.default_rng(1).standard_normal((50, D)).astype(np.float32)
    y32 = oracle.wht_rotate_fp32(u, s)
    assert y32.dtype == np.float32
    assert np.max(np.abs(y32 - u.astype(np.float64) @ R.T)) < 1e-5


def test_wht_signs_balanced():
    s = oracle.wht_signs(99, 1 << 14)
    assert abs(s.mean()) < 0.05


def test_fp32_rotation_constant():
    assert np.float32(1.0 / math.sqrt(D)).view(np.uint32) == 0x3DB504F3


@pytest.mark.parametrize("seed", [2, 3, 17])
def test_dense_rotation_is_q_of_gaussian_with_positive_r(seed):
    G = oracle.gaussian_matrix(seed, D, D)
    Pi = oracle.dense_rotation(seed, D)
    assert np.max(np.abs(Pi.T @ Pi - np.eye(D))) < 1e-13
    Rf = Pi.T @ G  # must be upper triangular with a positive diagonal (G = Pi R)
    assert np.max(np.abs(np.tril(Rf, -1))) < 1e-11
    assert np.all(np.diag(Rf) > 0)
    P32 = Pi.astype(np.float32).astype(np.float64)
    assert np.max(np.abs(P32.T @ P32 - np.eye(D))) <= 1e-6


def test_inner_product_identity():
    """<q, Pi^T y> = <Pi q, y> (rotate the query instead of every key), fp64."""
    rot = Rotation("dense", 2)
    rng = np.random.default_rng(3)
    q = rng.standard_normal((100, D))
    y = rng.standard_normal((100, D))
    lhs = np.sum(q * rot.inverse(y), axis=1)
    rhs = np.sum(rot.forward(q) * y, axis=1)
    assert np.max(np.abs(lhs - rhs) / (np.abs(lhs) + 1e-300)) < 1e-10
    rot_w = Rotation("wht", 0)
    lhs = np.sum(q * rot_w.inverse(y), axis=1)
    rhs = np.sum(rot_w.forward(q) * y, axis=1)
    assert np.max(np.abs(lhs - rhs)) < 1e-10


def test_gaussian_generator_distribution():
    g = oracle.gaussian_matrix(1003, 256, 256).ravel()
    assert stats.kstest(g, "norm").pvalue > 0.01
    assert abs(g.mean()) < 0.01 and abs(g.std() - 1.0) < 0.01


def test_qjl_matrix_independent_of_rotation_seed():
    S = oracle.qjl_matrix(1003, D)
    G = oracle.gaussian_matrix(3, D, D)
    assert abs(np.corrcoef(S.ravel(), G.ravel())[0, 1]) < 0.02


def test_rotated_coordinate_is_sphere_marginal():
    """Statistical (not a parity pin): for a fixed anisotropic x, coordinate 0 of Pi x/|x|
    over independent dense rotations follows the sphere marginal, (y+1)/2 ~ Beta((d-1)/2, (d-1)/2)."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal(D) * np.exp(rng.normal(0, 1.0, D))
    u = x / np.linalg.norm(x)
    ys = [(oracle.dense_rotation(seed, D) @ u)[0] for seed in range(1000, 1300)]
    a = (D - 1) / 2.0
    assert stats.kstest((np.array(ys) + 1) / 2, stats.beta(a, a).cdf).pvalue > 0.01
