"""Decode attention over a compressed KV cache (oracle; test infrastructure only).

Two routines:

* ``attention_reference`` -- the plain definition: dequantize every key and
  value in fp64, then scaled dot-product softmax attention with the maximum
  subtracted.  Rotating q once ([Triton deep dive] trick 1: <q, Pi y> =
  <Pi^T q, y> for orthogonal Pi) and online softmax ([Triton deep dive] trick 3:
  running m_i, l_i, acc rescaled by exp(m_old - m_new), one division at the end)
  are exact identities, so the fused GPU path must reach this result up to
  rounding.
* ``attention_compressed_domain`` -- the fused algebra written out in fp64:
  rotate q once (and sketch it once with S for QJL keys, [Triton deep dive]
  trick 2), score every key from its indices (n * <q_rot, c[idx]>, plus
  n * gamma * sqrt(pi/2)/d * <S q, sigma> for prod keys), run online softmax over
  key chunks, accumulate values in the rotated basis, merge the chunks, and
  un-rotate the output once.

Readings: scale = 1/sqrt(d) unless given ([turbo4 post-mortem] section 9: the
attention logit is q.k/sqrt(d)); no mask (decode attends every one of
seq_lens[b] keys); q-head h reads KV head floor(h * Hkv / Hq); turbo4 values are
rotated and quantized exactly like keys, so the rotated-basis accumulator is
un-rotated once per head (exact: sum_t p_t Pi^T y_t = Pi^T sum_t p_t y_t).
"""

import math

import numpy as np

from .formats import QJL_SCALE_NUM


def gqa_kv_head(h, Hq, Hkv):
    """KV head read by q-head h: consecutive q-heads share a KV head."""
    return (h * Hkv) // Hq


def attention_reference(q, k_hat, v_hat, seq_lens=None, scale=None):
    """Plain fp64 attention.

    q: [B, Hq, d]; k_hat, v_hat: [B, Hkv, L, d] dequantized keys and values.
    Returns (out [B, Hq, d], scores [B, Hq, L] with NaN beyond seq_lens[b]).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    Hkv, L = k_hat.shape[1], k_hat.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lens = [L] * B if seq_lens is None else list(seq_lens)
    out = np.zeros((B, Hq, d))
    scores = np.full((B, Hq, L), np.nan)
    for b in range(B):
        Lb = lens[b]
        for h in range(Hq):
            kv = gqa_kv_head(h, Hq, Hkv)
            s = (k_hat[b, kv, :Lb] @ q[b, h]) * scale
            p = np.exp(s - s.max())
            out[b, h] = (p / p.sum()) @ v_hat[b, kv, :Lb]
            scores[b, h, :Lb] = s
    return out, scores


def prefill_reference(q, k_hat, v_hat, q_start, scale=None):
    """Causal chunk attention, the prefill of [turbo4 post-mortem] section 9 (a prompt
    processed in chunks against the cache that already holds the chunk's own rows).

    q: [B, T, Hq, d]; k_hat, v_hat: [B, Hkv, L, d]; query i of sequence b sits at
    position q_start[b] + i.  Reading: the usual causal mask, keys at positions up to
    and including the query's own (the pages name the prefill but not its mask).  Each
    query is the plain definition of ``attention_reference`` over keys
    0 .. q_start[b] + i.  Returns out [B, T, Hq, d].
    """
    q = np.asarray(q, dtype=np.float64)
    B, T, Hq, d = q.shape
    out = np.zeros((B, T, Hq, d))
    for i in range(T):
        lens = [int(q_start[b]) + i + 1 for b in range(B)]
        out[:, i], _ = attention_reference(q[:, i], k_hat, v_hat, lens, scale)
    return out


def online_softmax_merge(partials):
    """Merge (m, l, acc) partials of one head by log-sum-exp rescaling.

    m* = max m_s, l* = sum l_s e^{m_s - m*}, acc* = sum acc_s e^{m_s - m*};
    empty partials (l = 0, m = -inf) are skipped.
    """
    live = [p for p in partials if p[1] > 0.0]
    m_star = max(p[0] for p in live)
    l_star = sum(p[1] * math.exp(p[0] - m_star) for p in live)
    acc = sum(p[2] * math.exp(p[0] - m_star) for p in live)
    return m_star, l_star, acc


def _chunk_partial(s, vals):
    """One online-softmax pass over a chunk of keys, block by block ([Triton deep dive] trick 3)."""
    m, l, acc = -math.inf, 0.0, np.zeros(vals.shape[1])
    for t in range(len(s)):
        m_new = max(m, s[t])
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        p = math.exp(s[t] - m_new)
        l = l * alpha + p
        acc = acc * alpha + p * vals[t]
        m = m_new
    return m, l, acc


def attention_compressed_domain(q, k_codec, k_blocks, v_codec, v_blocks, seq_lens=None,
                                scale=None, n_chunks=1):
    """Compressed-domain decode (fp64): rotate q once, score from indices, online softmax.

    q: [B, Hq, d]; k_blocks / v_blocks: packed rows [B, Hkv, L, row_bytes].
    Supported pairs: keys turbo4, turbo3 or prod3, values turbo4, turbo3 or vgroup2
    (turbo3 blocks and the blocks of d = 256 turbo4 rows carry per-block norms).
    Returns (out [B, Hq, d], scores [B, Hq, L]).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    Hkv, L = k_blocks.shape[1], k_blocks.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lens = [L] * B if seq_lens is None else list(seq_lens)
    out = np.zeros((B, Hq, d))
    scores = np.full((B, Hq, L), np.nan)
    for b in range(B):
        Lb = lens[b]
        for kv in range(Hkv):
            kf = k_codec.fields(k_blocks[b, kv, :Lb])
            vf = v_codec.fields(v_blocks[b, kv, :Lb])
            if "n_elem" in vf:  # per-block norms
                vals = vf["y_hat"] * vf["n_elem"]  # rotated basis
            elif v_codec.fmt == "turbo4":
                vals = vf["y_hat"] * vf["n"][:, None]  # rotated basis
            else:
                vals = vf["v_hat"]
            for h in range(Hq):
                if gqa_kv_head(h, Hq, Hkv) != kv:
                    continue
                q_rot = k_codec.rot.forward(q[b, h][None, :])[0]  # trick 1: once per query
                if "n_elem" in kf:  # per-block norms
                    s = (kf["y_hat"] * kf["n_elem"]) @ q_rot
                else:
                    s = kf["n"] * (kf["y_hat"] @ q_rot)
                if k_codec.fmt == "prod3":
                    q_sk = k_codec.S32.astype(np.float64) @ q[b, h]  # trick 2: once per query
                    s = s + kf["n"] * kf["gamma"] * k_codec.qjl_factor * (QJL_SCALE_NUM / d) * (kf["sigma"] @ q_sk)
                s = s * scale
                bounds = np.linspace(0, Lb, n_chunks + 1).astype(int)
                parts = [_chunk_partial(s[a:e], vals[a:e]) for a, e in zip(bounds[:-1], bounds[1:]) if e > a]
                _, l_star, acc = online_softmax_merge(parts)
                o = acc / l_star
                if v_codec.fmt in ("turbo4", "turbo3"):
                    o = v_codec.rot.inverse(o[None, :])[0]  # un-rotate once
                out[b, h] = o
                scores[b, h, :Lb] = s
    return out, scores
