"""Seeded random rotations and the QJL matrix (oracle; test infrastructure only).

Two rotations are used by the pages:

* randomized Hadamard / WHT: "WHT rotation" of the KV vectors before PolarQuant
  ([turbo4 post-mortem] sections 1, 2 bug 7, 10): y = (1/sqrt(d)) H D u with D a
  seeded +-1 diagonal and H the Sylvester Hadamard matrix, applied with the
  O(d log d) butterfly;
* a dense orthogonal Pi ([Triton deep dive] trick 1: keys are rotated with
  y = x @ Pi^T, Pi orthogonal, d x d), here the Q factor of the QR
  decomposition of a seeded Gaussian matrix.

The QJL stage projects with a Gaussian S that must be independent of the
rotation ([turbo4 post-mortem] section 10: correlated WHT/SRHT rotations broke
QJL; independent seeds fixed it).

Readings (the pages do not say how randomness is drawn): every random number
comes from the splitmix64 counter generator (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014): output i of seed s is
mix(s + (i + 1) * 0x9E3779B97F4A7C15).  WHT sign j is -1 when the top bit of
output j is set.  Gaussians use Box-Muller on consecutive output pairs.  The QR
factor is made unique by requiring diag(R) > 0.  Convention: y = Pi @ u
(column form; the row form x @ Pi^T of [Triton deep dive] is the same map) and
u = Pi^T @ y.  The query is rotated the same way as the keys.
"""

import math

import numpy as np

_MASK64 = (1 << 64) - 1
_GOLDEN_GAMMA = 0x9E3779B97F4A7C15


def splitmix64(seed, n, start=0):
    """Outputs start .. start+n-1 of splitmix64 seeded with ``seed`` (uint64 array).

    Output i is mix(seed + (i + 1) * gamma) with gamma = 0x9E3779B97F4A7C15 and
    mix(z) = z ^ (z >> 31) after z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9 and
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB, all modulo 2^64.
    """
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    z = np.uint64(seed & _MASK64) + i * np.uint64(_GOLDEN_GAMMA)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def wht_signs(seed, d):
    """The seeded +-1 diagonal D of the randomized Hadamard rotation (float64 array)."""
    top = splitmix64(seed, d) >> np.uint64(63)
    return np.where(top == 1, -1.0, 1.0)


def fwht(v):
    """Unnormalised fast Walsh-Hadamard transform along the last axis, H @ v.

    Stages h = 1, 2, 4, ..., d/2; for each i with (i & h) == 0 the pair becomes
    (v_i + v_{i+h}, v_i - v_{i+h}).  Works in the dtype of ``v`` (each stage is a
    separate rounded add/subtract), so fp32 input gives the canonical fp32
    sequence and fp64 input an fp64 transform.
    """
    v = np.array(v, copy=True)
    d = v.shape[-1]
    lead = v.shape[:-1]
    h = 1
    while h < d:
        w = v.reshape(lead + (d // (2 * h), 2, h))
        a = w[..., 0, :].copy()
        b = w[..., 1, :].copy()
        w[..., 0, :] = a + b
        w[..., 1, :] = a - b
        v = w.reshape(lead + (d,))
        h *= 2
    return v


def wht_rotate_fp32(u32, signs):
    """Canonical fp32 randomized-Hadamard rotation y = RN(1/sqrt(d)) * H (D u).

    Sign flips are exact, each butterfly stage is one rounded fp32 add or
    subtract, and the final scale is one rounded fp32 multiply by the fp32
    constant nearest 1/sqrt(d).
    """
    u32 = np.asarray(u32, dtype=np.float32)
    d = u32.shape[-1]
    v = u32 * signs.astype(np.float32)
    v = fwht(v)
    return (v * np.float32(1.0 / math.sqrt(d))).astype(np.float32)


def wht_rotation_matrix(signs):
    """Exact (fp64) matrix R = (1/sqrt(d)) H D of the randomized Hadamard rotation."""
    d = len(signs)
    H = fwht(np.eye(d, dtype=np.float64))  # columns H e_j; H is symmetric
    return H * signs[None, :] / math.sqrt(d)


def gaussian_matrix(seed, rows, cols):
    """rows x cols i.i.d. N(0,1) (fp64), row-major, Box-Muller on splitmix64 pairs.

    Pair p uses outputs 2p and 2p+1: u1 = ((o_2p >> 11) + 1) * 2^-53 in (0, 1],
    u2 = (o_2p+1 >> 11) * 2^-53 in [0, 1); r = sqrt(-2 ln u1); element 2p gets
    r cos(2 pi u2) and element 2p+1 gets r sin(2 pi u2).
    """
    n = rows * cols
    n_pairs = (n + 1) // 2
    raw = splitmix64(seed, 2 * n_pairs).tolist()
    out = np.empty(2 * n_pairs, dtype=np.float64)
    for p in range(n_pairs):
        u1 = ((raw[2 * p] >> 11) + 1) * (2.0 ** -53)
        u2 = (raw[2 * p + 1] >> 11) * (2.0 ** -53)
        r = math.sqrt(-2.0 * math.log(u1))
        out[2 * p] = r * math.cos(2.0 * math.pi * u2)
        out[2 * p + 1] = r * math.sin(2.0 * math.pi * u2)
    return out[:n].reshape(rows, cols)


def dense_rotation(seed, d):
    """Dense orthogonal Pi = Q of G = QR with diag(R) > 0, G = gaussian_matrix(seed) (fp64).

    [Triton deep dive] trick 1 (random orthogonal rotation of the keys).  The
    stored rotation used by both the encoder and attention is Pi rounded to fp32.
    """
    G = gaussian_matrix(seed, d, d)
    Q, R = np.linalg.qr(G)
    s = np.where(np.diag(R) < 0.0, -1.0, 1.0)
    return Q * s[None, :]


def qjl_matrix(seed, d):
    """QJL projection S (d x d, i.i.d. N(0,1), fp64) drawn from its own seed.

    [Triton deep dive] trick 2 uses a d x d S with the constant sqrt(pi/2)/d,
    i.e. N(0,1) entries; [turbo4 post-mortem] section 10 requires S to be
    independent of the rotation.
    """
    return gaussian_matrix(seed, d, d)
