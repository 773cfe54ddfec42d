"""Pins of the oracle's attention: the fused compressed-domain algebra against the plain
dequantize-then-softmax definition, plus special cases."""

import math

import numpy as np
import pytest

import oracle
from oracle.formats import Codec

D = 128

PAIRS = [
    ("turbo4", "turbo4", "wht"),
    ("turbo4", "turbo4", "dense"),
    ("prod3", "vgroup2", "dense"),
]


def make_cache(codec, B, Hkv, L, seed, scale=1.0):
    x = (np.random.default_rng(seed).standard_normal((B * Hkv * L, D)) * scale).astype(np.float32)
    blk, _ = codec.encode(x)
    return blk.reshape(B, Hkv, L, -1)


def dequant(codec, blocks):
    B, Hkv, L, rb = blocks.shape
    return codec.dequantize(blocks.reshape(-1, rb)).reshape(B, Hkv, L, D)


@pytest.mark.parametrize("kfmt,vfmt,rot", PAIRS)
def test_compressed_domain_equals_bruteforce(kfmt, vfmt, rot):
    """Rotate q once, score from indices, accumulate in the rotated basis, un-rotate once:
    equal to dequantize-then-softmax within 1e-10 (fp64) on tiny inputs."""
    B, Hq, Hkv, L = 2, 6, 2, 48
    kc = Codec(kfmt, rotation=rot, rot_seed=3, qjl_seed=1003)
    vc = Codec(vfmt, rotation=rot, rot_seed=4)
    kb = make_cache(kc, B, Hkv, L, 1, scale=2.0)
    vb = make_cache(vc, B, Hkv, L, 2)
    q = np.random.default_rng(3).standard_normal((B, Hq, D))
    lens = [37, 48]
    ref, s_ref = oracle.attention_reference(q, dequant(kc, kb), dequant(vc, vb), lens)
    out, s = oracle.attention_compressed_domain(q, kc, kb, vc, vb, lens, n_chunks=3)
    assert np.max(np.abs(out - ref)) < 1e-10
    m = ~np.isnan(s_ref)
    assert np.array_equal(m, ~np.isnan(s))
    assert np.max(np.abs(s[m] - s_ref[m])) < 1e-10


def test_prod_score_is_inner_product_with_reconstruction():
    """prod score = <q, x_hat>/sqrt(d) computed by brute force, to 1e-10."""
    kc = Codec("prod3", rotation="dense", rot_seed=3, qjl_seed=1003)
    vc = Codec("vgroup2")
    kb = make_cache(kc, 1, 1, 20, 5, scale=3.0)
    vb = make_cache(vc, 1, 1, 20, 6)
    q = np.random.default_rng(7).standard_normal((1, 1, D))
    _, s = oracle.attention_compressed_domain(q, kc, kb, vc, vb)
    xh = kc.dequantize(kb.reshape(-1, 56))
    assert np.max(np.abs(s[0, 0] - xh @ q[0, 0] / math.sqrt(D))) < 1e-10


def test_online_softmax_split_invariance():
    kc = Codec("turbo4", rotation="wht", rot_seed=0)
    kb = make_cache(kc, 1, 1, 64, 9)
    vb = make_cache(kc, 1, 1, 64, 10)
    q = np.random.default_rng(8).standard_normal((1, 2, D)) * 3
    one, _ = oracle.attention_compressed_domain(q, kc, kb, kc, vb, n_chunks=1)
    for n in (2, 5, 64):
        many, _ = oracle.attention_compressed_domain(q, kc, kb, kc, vb, n_chunks=n)
        assert np.max(np.abs(many - one)) < 1e-12


def test_merge_skips_empty_partials():
    acc = np.ones(3)
    m, l, a = oracle.online_softmax_merge([(-math.inf, 0.0, np.zeros(3)), (0.5, 2.0, acc)])
    assert m == 0.5 and l == 2.0 and np.array_equal(a, acc)


def test_uniform_scores_give_mean_of_values():
    """q = 0 makes every score equal, so the output is the plain mean of V_hat."""
    kc = Codec("turbo4", rotation="dense", rot_seed=1)
    kb = make_cache(kc, 1, 1, 33, 11)
    vb = make_cache(kc, 1, 1, 33, 12)
    q = np.zeros((1, 1, D))
    out, _ = oracle.attention_compressed_domain(q, kc, kb, kc, vb)
    assert np.allclose(out[0, 0], dequant(kc, vb)[0, 0].mean(axis=0), atol=1e-13)


def test_single_key_returns_its_value():
    kc = Codec("turbo4", rotation="wht", rot_seed=2)
    kb = make_cache(kc, 1, 1, 1, 13)
    vb = make_cache(kc, 1, 1, 1, 14)
    q = np.random.default_rng(1).standard_normal((1, 3, D))
    out, _ = oracle.attention_reference(q, dequant(kc, kb), dequant(kc, vb))
    assert np.allclose(out[0], dequant(kc, vb)[0, 0, 0][None, :], atol=1e-14)


def test_gqa_mapping_consecutive_heads():
    assert [oracle.gqa_kv_head(h, 32, 8) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.gqa_kv_head(h, 24, 4) for h in (5, 6, 23)] == [0, 1, 3]
    assert [oracle.gqa_kv_head(h, 4, 4) for h in range(4)] == [0, 1, 2, 3]


def test_reference_is_softmax_definition():
    """Two keys with a known score gap give the closed-form logistic weights."""
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = math.sqrt(D)  # score = k[0]
    k = np.zeros((1, 1, 2, D))
    k[0, 0, 0, 0], k[0, 0, 1, 0] = 1.0, 3.0
    v = np.zeros((1, 1, 2, D))
    v[0, 0, 0, 1], v[0, 0, 1, 1] = 1.0, 0.0
    out, s = oracle.attention_reference(q, k, v)
    assert np.allclose(s[0, 0], [1.0, 3.0])
    assert abs(out[0, 0, 1] - 1.0 / (1.0 + math.exp(2.0))) < 1e-15
