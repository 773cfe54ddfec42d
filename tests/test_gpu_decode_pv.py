"""GPU parity of the fused decode over prod3 keys (2-bit MSE + 1-bit QJL) and vgroup2
values (2-bit group codes) against the oracle.

Small shapes use caches encoded by the oracle, so both sides attend over identical
packed bytes: scores (max abs 2e-3) and outputs (max abs 2e-3, per-head relative 1e-3)
are compared element by element.  The full-size workload (B=4, Hq=24, Hkv=4, L=30,000)
runs with caches written by the GPU write path; sampled heads are checked against the
oracle run on those same packed bytes."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import ATOL, check_outputs, lib, torch_rows
from oracle.formats import Codec
from test_gpu_decode import upload_cache

pytestmark = pytest.mark.gpu

ROT_SEED, QJL_SEED = 3, 1003


def codecs():
    return Codec("prod3", rotation="dense", rot_seed=ROT_SEED, qjl_seed=QJL_SEED), Codec("vgroup2")


def contexts(tq):
    return tq.Ctx("prod3", "dense", ROT_SEED, QJL_SEED), tq.Ctx("vgroup2")


def encoded(codec, B, Hkv, L, seed, scale=1.0, lognormal=False):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((B * Hkv * L, 128)) * scale).astype(np.float32)
    if lognormal:
        s = np.exp(rng.normal(0, 0.5, 128)).astype(np.float32)
        s[rng.integers(128)] *= 8
        x = x * s
    blk, _ = codec.encode(x)
    return blk.reshape(B, Hkv, L, -1)


def run(tq, kctx, vctx, q_t, kc, vc, B, Hq, Hkv, L, lens=None, scores=True, staged=False, scale=0.0):
    import torch
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    sc = torch.full((B, Hq, L), float("nan"), dtype=torch.float32, device="cuda") if scores else None
    sl = None if lens is None else torch.tensor(np.asarray(lens, np.int32), device="cuda")
    if staged:
        tq.tq_decode_prepare_q(kctx, vctx, q_t, ws, B, Hq, Hkv, L, scale=scale)
        tq.tq_decode_partial(kctx, vctx, kc, vc, ws, B, Hq, Hkv, L, seq_lens=sl, scores=sc)
        tq.tq_decode_combine(kctx, vctx, out, ws, B, Hq, Hkv, L)
    else:
        tq.tq_decode_attention(kctx, vctx, q_t, kc, vc, out, ws, B, Hq, Hkv, L, seq_lens=sl, scores=sc,
                               scale=scale)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (sc.cpu().numpy() if scores else None)


def reference(q32, kcodec, kb, vcodec, vb, lens, scale=None):
    B, Hkv, L, _ = kb.shape
    kh = kcodec.dequantize(kb.reshape(-1, kb.shape[-1])).reshape(B, Hkv, L, 128)
    vh = vcodec.dequantize(vb.reshape(-1, vb.shape[-1])).reshape(B, Hkv, L, 128)
    return oracle.attention_reference(q32, kh, vh, lens, scale=scale)


CASES = [
    # B, Hq, Hkv, L, lens
    (2, 12, 2, 500, [300, 500]),      # 6 q-heads per KV head (the workload's ratio), ragged
    (1, 4, 1, 1000, None),            # 4 of the 8 head rows used, several tiles
    (1, 8, 1, 193, None),             # one full tile plus one key
    (2, 24, 2, 700, [1, 700]),        # 12 q-heads per KV head: two head groups; length 1
    (3, 6, 1, 64, [64, 5, 30]),       # shorter than one warp's share of a tile
]


@pytest.mark.parametrize("case", CASES)
def test_decode_prod3_vgroup2_parity(case):
    tq = lib()
    B, Hq, Hkv, L, lens = case
    kcodec, vcodec = codecs()
    kb = encoded(kcodec, B, Hkv, L, 21, scale=2.0, lognormal=True)
    vb = encoded(vcodec, B, Hkv, L, 22, scale=3.0)
    q_t, q32 = torch_rows(np.random.default_rng(23).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    kctx, vctx = contexts(tq)
    out, sc = run(tq, kctx, vctx, q_t, upload_cache(tq, "prod3", kb), upload_cache(tq, "vgroup2", vb),
                  B, Hq, Hkv, L, lens)
    ref, s_ref = reference(q32, kcodec, kb, vcodec, vb, lens)
    check_outputs(out, ref)
    m = ~np.isnan(s_ref)
    assert np.array_equal(m, ~np.isnan(sc)), "scores written for the wrong keys"
    assert np.max(np.abs(sc[m] - s_ref[m])) <= ATOL
    assert tq.tq_ctx_device_status(kctx) == 0


def test_decode_pv_peaked_attention_and_staged_calls():
    """A large scale makes the softmax peaked (a few keys carry the weight), which
    exposes any rounding of the probabilities; the staged calls give the same bits."""
    tq = lib()
    B, Hq, Hkv, L = 1, 6, 1, 900
    kcodec, vcodec = codecs()
    kb = encoded(kcodec, B, Hkv, L, 24, scale=3.0)
    vb = encoded(vcodec, B, Hkv, L, 25, scale=4.0)
    q_t, q32 = torch_rows(np.random.default_rng(26).standard_normal((B, Hq, 128)).astype(np.float32), "f32")
    kctx, vctx = contexts(tq)
    kc, vc = upload_cache(tq, "prod3", kb), upload_cache(tq, "vgroup2", vb)
    out1, _ = run(tq, kctx, vctx, q_t, kc, vc, B, Hq, Hkv, L, scores=False, scale=0.5)
    out2, _ = run(tq, kctx, vctx, q_t, kc, vc, B, Hq, Hkv, L, scores=False, staged=True, scale=0.5)
    ref, s = reference(q32, kcodec, kb, vcodec, vb, None, scale=0.5)
    assert np.nanmax(s) - np.nanmin(s) > 20  # genuinely peaked
    check_outputs(out1, ref)
    assert np.array_equal(out1, out2)


def test_decode_pv_constant_value_groups():
    """Groups whose values are all equal have scale 0: the output is carried by the zero
    points alone."""
    tq = lib()
    B, Hq, Hkv, L = 1, 6, 1, 300
    kcodec, vcodec = codecs()
    kb = encoded(kcodec, B, Hkv, L, 27)
    x = np.random.default_rng(28).standard_normal((L, 128)).astype(np.float32)
    x[:, 32:64] = 1.5    # one constant group in every row
    x[:100, :] = -0.25   # whole rows constant
    vb = vcodec.encode(x)[0].reshape(B, Hkv, L, -1)
    q_t, q32 = torch_rows(np.random.default_rng(29).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    kctx, vctx = contexts(tq)
    out, _ = run(tq, kctx, vctx, q_t, upload_cache(tq, "prod3", kb), upload_cache(tq, "vgroup2", vb),
                 B, Hq, Hkv, L, scores=False)
    ref, _ = reference(q32, kcodec, kb, vcodec, vb, None)
    check_outputs(out, ref)
    assert np.all(np.abs(out[..., 32:64] - ref[..., 32:64]) <= 1e-5 + ATOL)


def test_full_size_prod_vgroup():
    """B=4, Hq=24, Hkv=4, L=30,000: caches written by the GPU write path, decoded in the
    benchmark's launch configuration; sampled heads against the oracle on the same bytes."""
    import torch
    tq = lib()
    cfg = synth.WORKLOADS["prod_vgroup"]
    B, Hq, Hkv, L = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["L"]
    kctx, vctx = contexts(tq)
    kc, vc = tq.alloc_cache("prod3", B * Hkv * L), tq.alloc_cache("vgroup2", B * Hkv * L)
    for tensor, ctx, cache in (("K", kctx, kc), ("V", vctx, vc)):
        for b in range(B):
            for h in range(Hkv):
                _, bits = synth.kv_unit(cfg, tensor, b, h)
                src = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
                rows = torch.arange((b * Hkv + h) * L, (b * Hkv + h + 1) * L, dtype=torch.int64, device="cuda")
                tq.tq_quantize_set_rows(ctx, src, cache, row_ids=rows)
    q32, qbits = synth.queries(cfg)
    q_t = torch.from_numpy(qbits.view(np.int16)).view(torch.bfloat16).cuda()
    out, _ = run(tq, kctx, vctx, q_t, kc, vc, B, Hq, Hkv, L, scores=False)
    assert tq.tq_ctx_device_status(kctx) == 0
    kcodec, vcodec = codecs()
    khost, vhost = kc.cpu().numpy(), vc.cpu().numpy()
    for (b, h) in [(0, 0), (1, 11), (3, 23)]:
        kv = oracle.gqa_kv_head(h, Hq, Hkv)
        u = b * Hkv + kv
        kb = khost[u * L * 56:(u + 1) * L * 56].reshape(1, 1, L, 56)
        vb = vhost[u * L * 48:(u + 1) * L * 48].reshape(1, 1, L, 48)
        ref, _ = reference(q32[b:b + 1, h:h + 1], kcodec, kb, vcodec, vb, None)
        check_outputs(out[b:b + 1, h:h + 1], ref)


def test_decode_pv_many_heads_staged_prep():
    """1056 query heads (44 batches x 24) through the q preparation with the QJL sketch."""
    tq = lib()
    B, Hq, Hkv, L = 44, 24, 4, 40
    kcodec, vcodec = codecs()
    kb = encoded(kcodec, B, Hkv, L, 30)
    vb = encoded(vcodec, B, Hkv, L, 31)
    q_t, q32 = torch_rows(np.random.default_rng(32).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    kctx, vctx = contexts(tq)
    out, sc = run(tq, kctx, vctx, q_t, upload_cache(tq, "prod3", kb), upload_cache(tq, "vgroup2", vb),
                  B, Hq, Hkv, L)
    ref, s_ref = reference(q32, kcodec, kb, vcodec, vb, None)
    check_outputs(out, ref)
    assert np.max(np.abs(sc - s_ref)) <= ATOL


def test_decode_pv_shrunk_qjl_and_sphere_codebook():
    """The 2/pi-shrunk QJL term and the sphere-marginal 2-bit codebook: the same kernel
    with a different sketch scale and centroid table, against the oracle's estimator."""
    tq = lib()
    B, Hq, Hkv, L = 2, 12, 2, 333
    kcodec = Codec("prod3", rotation="dense", rot_seed=ROT_SEED, qjl_seed=QJL_SEED, codebook="sphere",
                   qjl_shrink=True)
    vcodec = Codec("vgroup2")
    kb = encoded(kcodec, B, Hkv, L, 41, scale=2.0, lognormal=True)
    vb = encoded(vcodec, B, Hkv, L, 42, scale=3.0)
    q_t, q32 = torch_rows(np.random.default_rng(43).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    kctx = tq.Ctx("prod3", "dense", ROT_SEED, QJL_SEED, codebook="sphere", qjl_shrink=True)
    vctx = tq.Ctx("vgroup2")
    out, sc = run(tq, kctx, vctx, q_t, upload_cache(tq, "prod3", kb), upload_cache(tq, "vgroup2", vb),
                  B, Hq, Hkv, L)
    ref, s_ref = reference(q32, kcodec, kb, vcodec, vb, None)
    check_outputs(out, ref)
    assert np.max(np.abs(sc - s_ref)) <= ATOL
    # the shrunk estimator really differs from the unbiased one on these bytes
    plain = Codec("prod3", rotation="dense", rot_seed=ROT_SEED, qjl_seed=QJL_SEED, codebook="sphere")
    ref_plain, _ = reference(q32, plain, kb, vcodec, vb, None)
    assert np.max(np.abs(ref_plain - ref)) > 10 * ATOL
