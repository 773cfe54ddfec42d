"""Pins of the oracle's causal chunk attention (prefill) against closed forms and
invariants that do not go through its own softmax code."""

import numpy as np

import oracle


def _inputs(B=2, T=6, Hq=4, Hkv=2, L=12, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, 8))
    k = rng.standard_normal((B, Hkv, L, 8))
    v = rng.standard_normal((B, Hkv, L, 8))
    return q, k, v


def test_identical_keys_give_prefix_means():
    """All keys equal: the softmax is uniform over the visible keys, so query i of
    sequence b returns the mean of values 0 .. q_start[b] + i (a running mean)."""
    q, k, v = _inputs()
    k[:] = k[:, :, :1]
    q_start = [0, 5]
    out = oracle.prefill_reference(q, k, v, q_start)
    for b in range(2):
        csum = np.cumsum(v[b], axis=1) / np.arange(1, v.shape[2] + 1)[None, :, None]
        for i in range(q.shape[1]):
            for h in range(4):
                kv = h * 2 // 4
                assert np.allclose(out[b, i, h], csum[kv, q_start[b] + i], atol=1e-12)


def test_first_query_of_a_sequence_sees_one_key():
    q, k, v = _inputs()
    out = oracle.prefill_reference(q, k, v, [0, 3])
    for h in range(4):
        assert np.allclose(out[0, 0, h], v[0, h * 2 // 4, 0], atol=1e-15)


def test_causality():
    """Changing keys or values after a query's position leaves it unchanged; changing the
    key at its own position changes it."""
    q, k, v = _inputs(seed=1)
    base = oracle.prefill_reference(q, k, v, [2, 4])
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 5] += 3.0
    v2[0, :, 5] -= 2.0
    out = oracle.prefill_reference(q, k2, v2, [2, 4])
    # sequence 0: query i at position 2 + i; positions 2, 3, 4 come before key 5
    assert np.array_equal(out[0, :3], base[0, :3])
    assert not np.allclose(out[0, 3], base[0, 3])
    assert np.array_equal(out[1], base[1])


def test_dominant_key():
    """A key far more aligned with the query than the others takes all the weight once
    it is visible, and none before."""
    q, k, v = _inputs(B=1, T=5, Hq=1, Hkv=1, L=9, seed=2)
    k[0, 0, 4] = 50.0 * q[0, 3, 0] / np.linalg.norm(q[0, 3, 0])
    out = oracle.prefill_reference(q, k, v, [1])  # query i at position 1 + i
    assert np.allclose(out[0, 3, 0], v[0, 0, 4], atol=1e-6)  # position 4: the key itself
    ref = oracle.attention_reference(q[:, 2], k[:, :, :4], v[:, :, :4])[0]
    assert np.allclose(out[0, 2], ref[0], atol=1e-15)  # position 3: the key is not yet visible
