"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds input generation only -- no step of the compression method.
Every array is drawn from numpy's ``default_rng`` with a seed sequence that
names the workload, the tensor and (for K/V caches) the (batch, KV-head) unit,
so any single unit can be regenerated cheaply by the oracle.

Workloads (shapes and distributions of the pages' decode and write workloads):

* ``single_head``: d=128, 512 keys/values + 1 query, fp32 N(0,1), seed 0,
  drawn in the order K, V, q.
* ``gqa_lognormal``: B=8, Hq=32, Hkv=8, L=32768; q bf16 N(0,1); K and V are
  N(0,1) times a per-(KV-head, channel) lognormal(0, 0.5) scale, with
  round(1% of 128) = 1 channel per KV head multiplied by 8 (chosen by a seeded
  permutation); separate draws for K and V; bf16; seed 2.
* ``prod_vgroup``: B=4, Hq=24, Hkv=4, L=30000; q bf16 N(0,1); K, V bf16 N(0,1);
  seed 3.
* ``write_chunk``: 16384 tokens x 8 KV heads x 128, bf16 N(0,1) K and V; seed 4.
* ``long_context``: B=1, Hq=32, Hkv=8, L=131072; bf16 q, K, V N(0,1); seed 5.
* ``gqa_t3k``: the ``gqa_lognormal`` recipe and seed unchanged (the same draws),
  for the asymmetric cache with 3-bit keys and 4-bit values.
* ``gqa_t3``: the same draws again, for the symmetric turbo3 cache (3-bit keys
  and values).
* ``gqa_d256``: head dimension 256 (turbo4): B=4, Hq=32, Hkv=8, L=32768, the
  ``gqa_lognormal`` law over 256 channels (round(1% of 256) = 3 outlier channels
  per KV head); seed 9.
* ``prefill_chunk``: B=1, Hq=32, Hkv=8, L=32768, T=512 chunk queries at positions
  L-T .. L-1 (the last chunk of a 32K-token prompt); K and V as ``gqa_lognormal``
  (lognormal channel scales with one outlier channel per KV head), bf16; q bf16
  N(0,1) [B, T, Hq, 128]; seed 7.

bf16 values are produced by rounding fp32 draws to nearest-even bf16; they are
returned both as uint16 bit patterns and as the exactly equal fp32 values.
"""

import zlib

import numpy as np

WORKLOADS = {
    "single_head": dict(B=1, Hq=1, Hkv=1, L=512, q_dtype="f32", kv_dtype="f32", dist="normal", seed=0),
    "gqa_lognormal": dict(B=8, Hq=32, Hkv=8, L=32768, q_dtype="bf16", kv_dtype="bf16", dist="lognormal_outlier", seed=2),
    "prod_vgroup": dict(B=4, Hq=24, Hkv=4, L=30000, q_dtype="bf16", kv_dtype="bf16", dist="normal", seed=3),
    "write_chunk": dict(N=16384, Hkv=8, kv_dtype="bf16", dist="normal", seed=4),
    "long_context": dict(B=1, Hq=32, Hkv=8, L=131072, q_dtype="bf16", kv_dtype="bf16", dist="normal", seed=5),
    # the gqa_lognormal recipe again, for the asymmetric 3-bit-key / 4-bit-value cache
    "gqa_t3k": dict(B=8, Hq=32, Hkv=8, L=32768, q_dtype="bf16", kv_dtype="bf16", dist="lognormal_outlier", seed=2),
    # and for the symmetric 3.5-bit cache (turbo3 keys and values)
    "gqa_t3": dict(B=8, Hq=32, Hkv=8, L=32768, q_dtype="bf16", kv_dtype="bf16", dist="lognormal_outlier", seed=2),
    # the last 512-token chunk of a 32K-token prompt: T chunk queries at positions L-T .. L-1
    "prefill_chunk": dict(B=1, Hq=32, Hkv=8, L=32768, T=512, q_dtype="bf16", kv_dtype="bf16",
                          dist="lognormal_outlier", seed=7),
    # head dimension 256: the gqa_lognormal law over 256 channels, half the batch
    "gqa_d256": dict(B=4, Hq=32, Hkv=8, L=32768, d=256, q_dtype="bf16", kv_dtype="bf16",
                     dist="lognormal_outlier", seed=9),
}

D = 128


def _tag(name):
    return zlib.crc32(name.encode())


def bf16_bits(x32):
    """Round fp32 to bf16 (nearest-even; NaN kept quiet) and return uint16 bit patterns."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    nan = np.isnan(np.ascontiguousarray(x32, dtype=np.float32))
    rounded = np.where(nan, (u >> np.uint32(16)) | np.uint32(0x40), rounded)
    return rounded.astype(np.uint16)


def bf16_to_f32(bits):
    """Exact fp32 value of bf16 bit patterns."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _maybe_bf16(x32, dtype):
    if dtype == "bf16":
        bits = bf16_bits(x32)
        return bf16_to_f32(bits), bits
    return np.asarray(x32, dtype=np.float32), None


def channel_scales(cfg, tensor):
    """Per-(KV-head, channel) multipliers [Hkv, 128] for the lognormal-with-outliers law."""
    rng = np.random.default_rng([cfg["seed"], _tag(tensor), _tag("scales")])
    d = cfg.get("d", D)
    s = np.exp(rng.normal(0.0, 0.5, size=(cfg["Hkv"], d)))
    n_out = int(round(0.01 * d))
    for h in range(cfg["Hkv"]):
        s[h, rng.permutation(d)[:n_out]] *= 8.0
    return s


def kv_unit(cfg, tensor, b, h, L=None):
    """K or V rows of one (batch, KV-head) unit: (fp32 values [L, 128], bf16 bits or None)."""
    L = cfg["L"] if L is None else L
    rng = np.random.default_rng([cfg["seed"], _tag(tensor), b, h])
    z = rng.standard_normal((L, cfg.get("d", D)), dtype=np.float32)
    if cfg["dist"] == "lognormal_outlier":
        z = (z * channel_scales(cfg, tensor)[h][None, :].astype(np.float32)).astype(np.float32)
    return _maybe_bf16(z, cfg["kv_dtype"])


def kv_cache_inputs(cfg, tensor, L=None):
    """All units: (fp32 [B, Hkv, L, 128], bf16 bits or None)."""
    L = cfg["L"] if L is None else L
    vals = np.empty((cfg["B"], cfg["Hkv"], L, D), dtype=np.float32)
    bits = np.empty((cfg["B"], cfg["Hkv"], L, D), dtype=np.uint16) if cfg["kv_dtype"] == "bf16" else None
    for b in range(cfg["B"]):
        for h in range(cfg["Hkv"]):
            v, bb = kv_unit(cfg, tensor, b, h, L)
            vals[b, h] = v
            if bits is not None:
                bits[b, h] = bb
    return vals, bits


def queries(cfg, B=None, Hq=None):
    """q [B, Hq, 128]: (fp32 values, bf16 bits or None)."""
    B = cfg["B"] if B is None else B
    Hq = cfg["Hq"] if Hq is None else Hq
    rng = np.random.default_rng([cfg["seed"], _tag("q")])
    return _maybe_bf16(rng.standard_normal((B, Hq, cfg.get("d", D)), dtype=np.float32), cfg["q_dtype"])


def prefill_queries(cfg):
    """Chunk queries q [B, T, Hq, 128]: (fp32 values, bf16 bits or None)."""
    rng = np.random.default_rng([cfg["seed"], _tag("q"), _tag("prefill")])
    x = rng.standard_normal((cfg["B"], cfg["T"], cfg["Hq"], D), dtype=np.float32)
    return _maybe_bf16(x, cfg["q_dtype"])


def single_head_inputs():
    """The single-head workload drawn in the order K, V, q from one stream (seed 0)."""
    rng = np.random.default_rng(0)
    K = rng.standard_normal((512, D)).astype(np.float32)
    V = rng.standard_normal((512, D)).astype(np.float32)
    q = rng.standard_normal((D,)).astype(np.float32)
    return K, V, q


def write_rows(cfg, tensor, n_tokens=None):
    """Rows to quantize for the write workload: [tokens * Hkv, 128] (fp32 values, bf16 bits)."""
    n_tokens = cfg["N"] if n_tokens is None else n_tokens
    rng = np.random.default_rng([cfg["seed"], _tag(tensor)])
    x = rng.standard_normal((n_tokens * cfg["Hkv"], D), dtype=np.float32)
    return _maybe_bf16(x, cfg["kv_dtype"])


def seq_lens(B, L, seed, ragged=True):
    """Per-batch lengths in [1, L] (the last one is L) for ragged-batch tests."""
    if not ragged:
        return np.full(B, L, dtype=np.int32)
    rng = np.random.default_rng([seed, _tag("seq_lens")])
    lens = rng.integers(1, L + 1, size=B).astype(np.int32)
    lens[-1] = L
    return lens


def row_permutation(n, seed):
    """A seeded permutation of cache slots for scatter (SET_ROWS) tests."""
    return np.random.default_rng([seed, _tag("rows")]).permutation(n).astype(np.int64)
