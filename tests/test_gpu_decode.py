"""GPU parity of the fused decode attention against the oracle.

Small shapes (several tiles, several splits, ragged tails and ragged batches) use
caches encoded by the oracle, so both sides attend over identical packed bytes and
scores can be compared one by one (max abs 2e-3) as well as outputs (max abs 2e-3,
per-head relative 1e-3).  The full-size workloads run in the launch configuration
the benchmark times, with caches written by the GPU write path, and compare sampled
heads against the oracle run on that head's own inputs."""

import math

import numpy as np
import pytest

import oracle
import synth
from gpu_util import ATOL, check_outputs, lib, torch_rows
from oracle.formats import Codec

pytestmark = pytest.mark.gpu


def oracle_cache(codec, B, Hkv, L, seed, scale=1.0, dist="normal"):
    x = (np.random.default_rng(seed).standard_normal((B * Hkv * L, 128)) * scale).astype(np.float32)
    if dist == "lognormal":
        s = np.exp(np.random.default_rng(seed + 1).normal(0, 0.5, 128)).astype(np.float32)
        s[7] *= 8
        x = x * s
    blk, _ = codec.encode(x)
    return blk.reshape(B, Hkv, L, -1)


def upload_cache(tq, fmt, blocks):
    import torch
    flat = blocks.reshape(-1)
    t = tq.alloc_cache(fmt, blocks.shape[0] * blocks.shape[1] * blocks.shape[2])
    t[: flat.size].copy_(torch.from_numpy(flat.copy()))
    return t


def run_decode(tq, kctx, vctx, q_t, kc, vc, B, Hq, Hkv, L, lens=None, scores=True, staged=False):
    import torch
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    sc = torch.full((B, Hq, L), float("nan"), dtype=torch.float32, device="cuda") if scores else None
    sl = None if lens is None else torch.tensor(np.asarray(lens, np.int32), device="cuda")
    if staged:
        tq.tq_decode_prepare_q(kctx, vctx, q_t, ws, B, Hq, Hkv, L)
        tq.tq_decode_partial(kctx, vctx, kc, vc, ws, B, Hq, Hkv, L, seq_lens=sl, scores=sc)
        tq.tq_decode_combine(kctx, vctx, out, ws, B, Hq, Hkv, L)
    else:
        tq.tq_decode_attention(kctx, vctx, q_t, kc, vc, out, ws, B, Hq, Hkv, L, seq_lens=sl, scores=sc)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (sc.cpu().numpy() if scores else None)


def reference(q32, kcodec, kb, vcodec, vb, lens):
    B, Hkv, L, _ = kb.shape
    kh = kcodec.dequantize(kb.reshape(-1, kb.shape[-1])).reshape(B, Hkv, L, 128)
    vh = vcodec.dequantize(vb.reshape(-1, vb.shape[-1])).reshape(B, Hkv, L, 128)
    return oracle.attention_reference(q32, kh, vh, lens)


CASES = [
    # B, Hq, Hkv, L, lens
    (2, 8, 2, 300, [137, 300]),       # GQA 4, ragged batch, ragged tail, 2 splits
    (1, 1, 1, 512, None),             # single head
    (3, 6, 1, 1000, [1, 999, 1000]),  # GQA 6, a length-1 sequence
    (1, 12, 1, 700, None),            # 12 q-heads per KV head: two head groups
    (2, 8, 8, 129, [64, 129]),        # no grouping
]


@pytest.mark.parametrize("rot", ["wht", "dense"])
@pytest.mark.parametrize("case", CASES)
def test_decode_turbo4_parity(rot, case):
    tq = lib()
    B, Hq, Hkv, L, lens = case
    kcodec = Codec("turbo4", rotation=rot, rot_seed=3)
    vcodec = Codec("turbo4", rotation=rot, rot_seed=4)
    kb = oracle_cache(kcodec, B, Hkv, L, 1, scale=2.0, dist="lognormal")
    vb = oracle_cache(vcodec, B, Hkv, L, 2)
    q_t, q32 = torch_rows(np.random.default_rng(3).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    kctx, vctx = tq.Ctx("turbo4", rot, 3), tq.Ctx("turbo4", rot, 4)
    out, sc = run_decode(tq, kctx, vctx, q_t, upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb),
                         B, Hq, Hkv, L, lens)
    ref, s_ref = reference(q32, kcodec, kb, vcodec, vb, lens)
    check_outputs(out, ref)
    m = ~np.isnan(s_ref)
    assert np.array_equal(m, ~np.isnan(sc)), "scores written for the wrong keys"
    assert np.max(np.abs(sc[m] - s_ref[m])) <= ATOL
    assert tq.tq_ctx_device_status(kctx) == 0


@pytest.mark.parametrize("rot", ["wht", "dense"])
@pytest.mark.parametrize("case", CASES)
def test_decode_turbo3_keys_turbo4_values_parity(rot, case):
    """The asymmetric cache: 3-bit (2+1 layout) keys, 4-bit values."""
    tq = lib()
    B, Hq, Hkv, L, lens = case
    kcodec = Codec("turbo3", rotation=rot, rot_seed=13)
    vcodec = Codec("turbo4", rotation=rot, rot_seed=14)
    kb = oracle_cache(kcodec, B, Hkv, L, 11, scale=2.0, dist="lognormal")
    vb = oracle_cache(vcodec, B, Hkv, L, 12)
    q_t, q32 = torch_rows(np.random.default_rng(13).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    kctx, vctx = tq.Ctx("turbo3", rot, 13), tq.Ctx("turbo4", rot, 14)
    out, sc = run_decode(tq, kctx, vctx, q_t, upload_cache(tq, "turbo3", kb), upload_cache(tq, "turbo4", vb),
                         B, Hq, Hkv, L, lens)
    ref, s_ref = reference(q32, kcodec, kb, vcodec, vb, lens)
    check_outputs(out, ref)
    m = ~np.isnan(s_ref)
    assert np.array_equal(m, ~np.isnan(sc)), "scores written for the wrong keys"
    assert np.max(np.abs(sc[m] - s_ref[m])) <= ATOL
    assert tq.tq_ctx_device_status(kctx) == 0


@pytest.mark.parametrize("kfmt", ["turbo3", "turbo4"])
@pytest.mark.parametrize("rot", ["wht", "dense"])
@pytest.mark.parametrize("case", CASES)
def test_decode_turbo3_values_parity(kfmt, rot, case):
    """turbo3 values (3.5-bit, the 2+1 layout) with turbo3 keys (the symmetric turbo3 cache)
    or turbo4 keys."""
    tq = lib()
    B, Hq, Hkv, L, lens = case
    kcodec = Codec(kfmt, rotation=rot, rot_seed=33)
    vcodec = Codec("turbo3", rotation=rot, rot_seed=34)
    kb = oracle_cache(kcodec, B, Hkv, L, 31, scale=2.0, dist="lognormal")
    vb = oracle_cache(vcodec, B, Hkv, L, 32)
    q_t, q32 = torch_rows(np.random.default_rng(33).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    kctx, vctx = tq.Ctx(kfmt, rot, 33), tq.Ctx("turbo3", rot, 34)
    out, sc = run_decode(tq, kctx, vctx, q_t, upload_cache(tq, kfmt, kb), upload_cache(tq, "turbo3", vb),
                         B, Hq, Hkv, L, lens)
    ref, s_ref = reference(q32, kcodec, kb, vcodec, vb, lens)
    check_outputs(out, ref)
    m = ~np.isnan(s_ref)
    assert np.array_equal(m, ~np.isnan(sc)), "scores written for the wrong keys"
    assert np.max(np.abs(sc[m] - s_ref[m])) <= ATOL
    assert tq.tq_ctx_device_status(kctx) == 0


def test_decode_turbo3_values_own_block_norms():
    """Every 32-element value block is scaled by its own stored norm: blocks whose norms
    differ by up to 4x (and some set to zero) decode as the oracle's per-block
    dequantization says, with peaked attention (queries 2x) so few keys dominate; staged
    calls and 8 q-heads per KV head too."""
    tq = lib()
    B, Hq, Hkv, L = 2, 16, 2, 531
    kcodec = Codec("turbo3", rotation="wht", rot_seed=41)
    vcodec = Codec("turbo3", rotation="wht", rot_seed=42)
    kb = oracle_cache(kcodec, B, Hkv, L, 41)
    vb = oracle_cache(vcodec, B, Hkv, L, 42).copy()
    rng = np.random.default_rng(43)
    for c in range(4):
        n = vb[..., 14 * c:14 * c + 2].copy().view("<f2").astype(np.float32)
        f = rng.uniform(0.5, 2.0, size=n.shape).astype(np.float32)
        f[rng.random(n.shape) < 0.02] = 0.0
        vb[..., 14 * c:14 * c + 2] = (n * f).astype("<f2").view(np.uint8)
    q_t, q32 = torch_rows(rng.standard_normal((B, Hq, 128)).astype(np.float32) * 2.0, "f32")
    kctx, vctx = tq.Ctx("turbo3", "wht", 41), tq.Ctx("turbo3", "wht", 42)
    kc, vc = upload_cache(tq, "turbo3", kb), upload_cache(tq, "turbo3", vb)
    ref, s_ref = reference(q32, kcodec, kb, vcodec, vb, None)
    for staged in (False, True):
        out, sc = run_decode(tq, kctx, vctx, q_t, kc, vc, B, Hq, Hkv, L, staged=staged)
        check_outputs(out, ref)
        assert np.max(np.abs(sc - s_ref)) <= ATOL
    assert tq.tq_ctx_device_status(kctx) == 0


def test_decode_turbo3_keys_own_block_norms():
    """Every 32-element key block is scaled by its own stored norm: blocks whose norms
    differ (set here to other fp16 values, including zero) decode as the oracle's
    per-block dequantization says.  Staged calls, f32 queries, 8 q-heads per KV head."""
    tq = lib()
    B, Hq, Hkv, L = 2, 16, 2, 531
    kcodec = Codec("turbo3", rotation="wht", rot_seed=21)
    vcodec = Codec("turbo4", rotation="wht", rot_seed=22)
    kb = oracle_cache(kcodec, B, Hkv, L, 21).copy()
    vb = oracle_cache(vcodec, B, Hkv, L, 22)
    rng = np.random.default_rng(23)
    for c in range(4):
        n = kb[..., 14 * c:14 * c + 2].copy().view("<f2").astype(np.float32)
        f = rng.uniform(0.25, 4.0, size=n.shape).astype(np.float32)
        f[rng.random(n.shape) < 0.02] = 0.0
        kb[..., 14 * c:14 * c + 2] = (n * f).astype("<f2").view(np.uint8)
    q_t, q32 = torch_rows(rng.standard_normal((B, Hq, 128)).astype(np.float32) * 1.5, "f32")
    kctx, vctx = tq.Ctx("turbo3", "wht", 21), tq.Ctx("turbo4", "wht", 22)
    out, sc = run_decode(tq, kctx, vctx, q_t, upload_cache(tq, "turbo3", kb), upload_cache(tq, "turbo4", vb),
                         B, Hq, Hkv, L, staged=True)
    ref, s_ref = reference(q32, kcodec, kb, vcodec, vb, None)
    check_outputs(out, ref)
    assert np.max(np.abs(sc - s_ref)) <= ATOL
    assert tq.tq_ctx_device_status(kctx) == 0


@pytest.mark.parametrize("q_dtype", ["f32", "bf16", "f16"])
def test_decode_q_dtypes_and_staged_calls(q_dtype):
    tq = lib()
    B, Hq, Hkv, L = 2, 4, 1, 257
    codec = Codec("turbo4", rotation="wht", rot_seed=0)
    kb, vb = oracle_cache(codec, B, Hkv, L, 5), oracle_cache(codec, B, Hkv, L, 6)
    q_t, q32 = torch_rows(np.random.default_rng(4).standard_normal((B, Hq, 128)).astype(np.float32), q_dtype)
    ctx = tq.Ctx("turbo4", "wht", 0)
    kc, vc = upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb)
    out1, _ = run_decode(tq, ctx, ctx, q_t, kc, vc, B, Hq, Hkv, L, scores=False)
    out2, _ = run_decode(tq, ctx, ctx, q_t, kc, vc, B, Hq, Hkv, L, scores=False, staged=True)
    ref, _ = reference(q32, codec, kb, codec, vb, None)
    check_outputs(out1, ref)
    # the one-call API merges the splits inside the split-K kernel: same arithmetic as the
    # combine kernel in another fp32 summation order
    np.testing.assert_allclose(out1, out2, rtol=2e-6, atol=1e-7)


def test_decode_many_heads_staged_kernels():
    """1152 query heads (36 batches x 32): many CTAs of the q-preparation and combine
    kernels, each serving eight heads."""
    tq = lib()
    B, Hq, Hkv, L = 36, 32, 8, 70
    codec = Codec("turbo4", rotation="dense", rot_seed=7)
    kb, vb = oracle_cache(codec, B, Hkv, L, 13), oracle_cache(codec, B, Hkv, L, 14)
    q_t, q32 = torch_rows(np.random.default_rng(8).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    ctx = tq.Ctx("turbo4", "dense", 7)
    out, sc = run_decode(tq, ctx, ctx, q_t, upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb),
                         B, Hq, Hkv, L)
    ref, s_ref = reference(q32, codec, kb, codec, vb, None)
    check_outputs(out, ref)
    assert np.max(np.abs(sc - s_ref)) <= ATOL


def test_decode_scale_argument_and_peaked_attention():
    """A large explicit scale makes the softmax peaked; results still match."""
    tq = lib()
    B, Hq, Hkv, L = 1, 4, 1, 400
    codec = Codec("turbo4", rotation="dense", rot_seed=1)
    kb, vb = oracle_cache(codec, B, Hkv, L, 7, scale=3.0), oracle_cache(codec, B, Hkv, L, 8)
    q_t, q32 = torch_rows(np.random.default_rng(5).standard_normal((B, Hq, 128)).astype(np.float32), "f32")
    ctx = tq.Ctx("turbo4", "dense", 1)
    import torch
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(ctx, ctx, B, Hq, Hkv, L))
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    scale = 0.5
    tq.tq_decode_attention(ctx, ctx, q_t, upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb), out, ws,
                           B, Hq, Hkv, L, scale=scale)
    kh = codec.dequantize(kb.reshape(-1, 68)).reshape(B, Hkv, L, 128)
    vh = codec.dequantize(vb.reshape(-1, 68)).reshape(B, Hkv, L, 128)
    ref, s = oracle.attention_reference(q32, kh, vh, scale=scale)
    assert np.nanmax(s) - np.nanmin(s) > 20  # genuinely peaked
    check_outputs(out.cpu().numpy(), ref)


def test_decode_zero_query_and_zero_values():
    """q = 0 gives uniform weights (mean of V_hat); all-zero value vectors give 0."""
    tq = lib()
    B, Hq, Hkv, L = 1, 2, 1, 200
    codec = Codec("turbo4", rotation="wht", rot_seed=2)
    kb = oracle_cache(codec, B, Hkv, L, 9)
    vb = oracle_cache(codec, B, Hkv, L, 10)
    vb_zero, _ = codec.encode(np.zeros((L, 128), np.float32))
    vb[0, 0, 100:] = vb_zero[100:]
    q = np.zeros((B, Hq, 128), np.float32)
    q[0, 1] = np.random.default_rng(1).standard_normal(128)
    q_t, q32 = torch_rows(q, "f32")
    ctx = tq.Ctx("turbo4", "wht", 2)
    out, _ = run_decode(tq, ctx, ctx, q_t, upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb),
                        B, Hq, Hkv, L, scores=False)
    ref, _ = reference(q32, codec, kb, codec, vb, None)
    check_outputs(out, ref)
    vh = codec.dequantize(vb.reshape(-1, 68))
    assert np.allclose(out[0, 0], vh.mean(0), atol=1e-5)


def test_decode_bad_seq_len_is_clamped_and_flagged():
    tq = lib()
    B, Hq, Hkv, L = 2, 2, 1, 100
    codec = Codec("turbo4", rotation="wht", rot_seed=0)
    kb, vb = oracle_cache(codec, B, Hkv, L, 11), oracle_cache(codec, B, Hkv, L, 12)
    q_t, q32 = torch_rows(np.random.default_rng(6).standard_normal((B, Hq, 128)).astype(np.float32), "f32")
    ctx = tq.Ctx("turbo4", "wht", 0)
    out, _ = run_decode(tq, ctx, ctx, q_t, upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb),
                        B, Hq, Hkv, L, lens=[500, 0], scores=False)
    assert tq.tq_ctx_device_status(ctx) == 2
    ref, _ = reference(q32, codec, kb, codec, vb, [100, 1])
    check_outputs(out, ref)


def test_decode_rejects_bad_arguments():
    import torch
    tq = lib()
    ctx = tq.Ctx("turbo4", "wht", 0)
    ws_small = tq.alloc_workspace(256)
    q = torch.zeros((1, 4, 128), dtype=torch.float32, device="cuda")
    cache = tq.alloc_cache("turbo4", 64)
    out = torch.zeros((1, 4, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention(ctx, ctx, q, cache, cache, out, ws_small, 1, 4, 1, 64)
    assert e.value.status == tq.TQ_ERR_WORKSPACE
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_workspace_size(ctx, ctx, 1, 5, 2, 64)  # Hq not a multiple of Hkv
    assert e.value.status == tq.TQ_ERR_INVALID_ARG
    t3, vg = tq.Ctx("turbo3", "wht", 0), tq.Ctx("vgroup2")
    for kc_, vc_ in ((t3, vg), (ctx, vg), (vg, ctx)):  # pairs without a decode kernel
        with pytest.raises(tq.TQError) as e:
            tq.tq_decode_workspace_size(kc_, vc_, 1, 4, 1, 64)
        assert e.value.status == tq.TQ_ERR_UNSUPPORTED


def _units(cfg, tensor, workers=16):
    """(b, h, bf16 bits) of every unit, drawn by a few host threads at a time."""
    from concurrent.futures import ThreadPoolExecutor
    units = [(b, h) for b in range(cfg["B"]) for h in range(cfg["Hkv"])]
    with ThreadPoolExecutor(max_workers=workers) as ex:
        for i in range(0, len(units), workers):
            chunk = units[i:i + workers]
            for (b, h), (_, bits) in zip(chunk, ex.map(lambda u: synth.kv_unit(cfg, tensor, *u), chunk)):
                yield b, h, bits


def _full_size(name, rot, rot_seed, sample_heads, k_fmt="turbo4", v_fmt="turbo4", **override):
    """Write the whole cache with the GPU write path, decode in the benchmark's launch
    configuration, and compare sampled (b, h) outputs with the oracle on that head's inputs."""
    import torch
    tq = lib()
    cfg = dict(synth.WORKLOADS[name], **override)
    B, Hq, Hkv, L = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["L"]
    kctx, vctx = tq.Ctx(k_fmt, rot, rot_seed), tq.Ctx(v_fmt, rot, rot_seed + 100)
    kc, vc = tq.alloc_cache(k_fmt, B * Hkv * L), tq.alloc_cache(v_fmt, B * Hkv * L)
    for tensor, ctx, cache in (("K", kctx, kc), ("V", vctx, vc)):
        for b, h, bits in _units(cfg, tensor):
            src = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
            rows = torch.arange((b * Hkv + h) * L, (b * Hkv + h + 1) * L, dtype=torch.int64, device="cuda")
            tq.tq_quantize_set_rows(ctx, src, cache, row_ids=rows)
    q32, qbits = synth.queries(cfg)
    q_t = torch.from_numpy(qbits.view(np.int16)).view(torch.bfloat16).cuda()
    out, _ = run_decode(tq, kctx, vctx, q_t, kc, vc, B, Hq, Hkv, L, scores=False)
    assert tq.tq_ctx_device_status(kctx) == 0
    kcod = Codec(k_fmt, rotation=rot, rot_seed=rot_seed)
    vcod = Codec(v_fmt, rotation=rot, rot_seed=rot_seed + 100)
    for (b, h) in sample_heads:
        kv = oracle.gqa_kv_head(h, Hq, Hkv)
        xk, _ = synth.kv_unit(cfg, "K", b, kv)
        xv, _ = synth.kv_unit(cfg, "V", b, kv)
        kh = kcod.dequantize(kcod.encode(xk)[0])[None, None]
        vh = vcod.dequantize(vcod.encode(xv)[0])[None, None]
        ref, _ = oracle.attention_reference(q32[b:b + 1, h:h + 1], kh, vh)
        check_outputs(out[b:b + 1, h:h + 1], ref)


def test_full_size_gqa_lognormal_dense():
    _full_size("gqa_lognormal", "dense", 2, [(0, 0), (3, 13), (7, 31)])


def test_full_size_long_context_wht():
    _full_size("long_context", "wht", 5, [(0, 0), (0, 17), (0, 31)])


def test_full_size_long_context_batch16_wht():
    """The largest point of the context sweep: B = 16 sequences of 131,072 keys (2.28 GB of
    packed K and V), sampled heads of the first, a middle and the last sequence."""
    _full_size("long_context", "wht", 5, [(0, 0), (7, 9), (15, 31)], B=16)


def test_full_size_gqa_turbo3_keys_and_values():
    _full_size("gqa_t3", "dense", 8, [(0, 0), (5, 18), (7, 31)], k_fmt="turbo3", v_fmt="turbo3")


def test_full_size_gqa_turbo3_keys():
    _full_size("gqa_t3k", "dense", 6, [(0, 0), (4, 21), (7, 31)], k_fmt="turbo3")


def test_decode_one_unit_many_splits():
    """One (batch, KV head) unit of 200,000 keys spread over every SM: about a hundred
    splits per head to merge, 8 q-heads per KV head (two column groups), a ragged last
    tile; all heads against the oracle on the GPU-written packed bytes."""
    import torch
    tq = lib()
    B, Hq, Hkv, L = 1, 8, 1, 200_000
    assert tq.tq_decode_num_splits(tq.Ctx("turbo4", "dense", 9), tq.Ctx("turbo4", "dense", 109), B, Hq, Hkv, L) > 50
    kctx, vctx = tq.Ctx("turbo4", "dense", 9), tq.Ctx("turbo4", "dense", 109)
    rng = np.random.default_rng(41)
    caches = []
    for ctx in (kctx, vctx):
        x = rng.standard_normal((L, 128), dtype=np.float32)
        t = torch.from_numpy(synth.bf16_bits(x).view(np.int16)).view(torch.bfloat16).cuda()
        cache = tq.alloc_cache("turbo4", L)
        tq.tq_quantize_set_rows(ctx, t, cache)
        caches.append(cache)
    q_t, q32 = torch_rows(rng.standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    out, _ = run_decode(tq, kctx, vctx, q_t, caches[0], caches[1], B, Hq, Hkv, L, scores=False)
    assert tq.tq_ctx_device_status(kctx) == 0
    kcod, vcod = Codec("turbo4", rotation="dense", rot_seed=9), Codec("turbo4", rotation="dense", rot_seed=109)
    kb = to_host_bytes_rows(caches[0], L).reshape(1, 1, L, 68)
    vb = to_host_bytes_rows(caches[1], L).reshape(1, 1, L, 68)
    ref, _ = reference(q32, kcod, kb, vcod, vb, None)
    check_outputs(out, ref)


def to_host_bytes_rows(cache, n):
    return cache.cpu().numpy()[: n * 68].reshape(n, 68)


def test_decode_shape_limits():
    """L = 0 and B = 0 are invalid; a shape whose tile count overflows 32 bits is refused."""
    tq = lib()
    ctx = tq.Ctx("turbo4", "wht", 0)
    for args in ((1, 4, 1, 0), (0, 4, 1, 64)):
        with pytest.raises(tq.TQError) as e:
            tq.tq_decode_workspace_size(ctx, ctx, *args)
        assert e.value.status == tq.TQ_ERR_INVALID_ARG
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_workspace_size(ctx, ctx, 1 << 20, 8, 8, 1 << 20)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("kfmt", ["turbo4", "turbo3"])
def test_decode_sphere_codebook(kfmt):
    """Sphere-marginal codebooks for keys and values: the kernels take any symmetric table."""
    tq = lib()
    B, Hq, Hkv, L = 2, 8, 2, 450
    kcodec = Codec(kfmt, rotation="wht", rot_seed=51, codebook="sphere")
    vcodec = Codec("turbo4", rotation="wht", rot_seed=52, codebook="sphere")
    kb = oracle_cache(kcodec, B, Hkv, L, 51, scale=2.0, dist="lognormal")
    vb = oracle_cache(vcodec, B, Hkv, L, 52)
    q_t, q32 = torch_rows(np.random.default_rng(53).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    kctx = tq.Ctx(kfmt, "wht", 51, codebook="sphere")
    vctx = tq.Ctx("turbo4", "wht", 52, codebook="sphere")
    out, sc = run_decode(tq, kctx, vctx, q_t, upload_cache(tq, kfmt, kb), upload_cache(tq, "turbo4", vb),
                         B, Hq, Hkv, L)
    ref, s_ref = reference(q32, kcodec, kb, vcodec, vb, None)
    check_outputs(out, ref)
    assert np.max(np.abs(sc - s_ref)) <= ATOL


@pytest.mark.parametrize("B,Hq,Hkv,L,fused", [(2, 8, 2, 300, True), (1, 8, 1, 60_000, True),
                                              (256, 8, 8, 240, False)])
def test_decode_merge_in_split_kernel_matches_combine(B, Hq, Hkv, L, fused):
    """tq_decode_attention lets the CTA that completes a unit merge its splits and write the
    outputs (two launches) unless CTAs would complete too many units (three launches, the
    combine kernel); either way the outputs equal the stage-by-stage path's (prepare_q,
    partial, combine) up to fp32 summation order, and the oracle's."""
    tq = lib()
    kcodec = Codec("turbo4", rotation="dense", rot_seed=13)
    vcodec = Codec("turbo4", rotation="dense", rot_seed=14)
    lens = list(np.random.default_rng(7).integers(1, L + 1, B)) if B > 1 else None
    kb = oracle_cache(kcodec, B, Hkv, L, 5, scale=2.0, dist="lognormal")
    vb = oracle_cache(vcodec, B, Hkv, L, 6)
    q_t, q32 = torch_rows(np.random.default_rng(8).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    kctx, vctx = tq.Ctx("turbo4", "dense", 13), tq.Ctx("turbo4", "dense", 14)
    assert tq.tq_decode_num_launches(kctx, vctx, B, Hq, Hkv, L) == (2 if fused else 3)
    kc, vc = upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb)
    for _ in range(2):  # twice: the unit counters are reset between calls
        out, _ = run_decode(tq, kctx, vctx, q_t, kc, vc, B, Hq, Hkv, L, lens, scores=False)
    staged, _ = run_decode(tq, kctx, vctx, q_t, kc, vc, B, Hq, Hkv, L, lens, scores=False, staged=True)
    np.testing.assert_allclose(out, staged, rtol=1e-5, atol=1e-6)
    # tq_decode_partial_merge repeated over one q preparation gives the same outputs
    import torch
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    sl = None if lens is None else torch.tensor(np.asarray(lens, np.int32), device="cuda")
    tq.tq_decode_prepare_q(kctx, vctx, q_t, ws, B, Hq, Hkv, L)
    for _ in range(3):
        merged = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        tq.tq_decode_partial_merge(kctx, vctx, kc, vc, merged, ws, B, Hq, Hkv, L, seq_lens=sl)
        # (the CTA completing a unit can differ between runs, and with it the merge's
        # fp32 summation order)
        np.testing.assert_allclose(merged.cpu().numpy(), out, rtol=1e-5, atol=1e-6)
    ref, _ = reference(q32, kcodec, kb, vcodec, vb, lens)
    check_outputs(out, ref)
    assert tq.tq_ctx_device_status(kctx) == 0


def test_decode_num_launches_prod3():
    """prod3 keys with vgroup2 values keep the combine kernel."""
    tq = lib()
    kctx, vctx = tq.Ctx("prod3", "dense", 1, 1001), tq.Ctx("vgroup2")
    assert tq.tq_decode_num_launches(kctx, vctx, 2, 12, 2, 1000) == 3
