"""GPU parity at head dimension 256 (turbo4 keys and values) against the oracle.

A 256-element row is rotated as a whole and stored as two 68-byte turbo4 blocks: the
randomized-Hadamard write is bit-exact against the oracle's canonical fp32 sequence, the
dense write agrees up to the 1e-5 boundary band, and the fused decode (rotate q once,
score from the indices with each block's own norm, online softmax split over CTAs, one
un-rotation) agrees with dequantize-then-softmax within the decode tolerances."""

import numpy as np
import pytest

import oracle
from gpu_util import band_ok, check_outputs, lib, torch_rows
from oracle.formats import Codec

pytestmark = pytest.mark.gpu

D2 = 256


def rows(n, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal((n, D2)) * scale).astype(np.float32)


def host_rows(cache, n):
    return cache.cpu().numpy()[: n * 136].reshape(n, 136)


@pytest.mark.parametrize("src", ["bf16", "f32"])
def test_write_wht_bit_exact(src):
    import torch
    tq = lib()
    n = 1000
    x_t, x32 = torch_rows(rows(n, 1, 3.0), src)
    ctx = tq.Ctx("turbo4", "wht", 5, d=D2)
    slots = np.random.default_rng(2).permutation(n + 37)[:n].astype(np.int64)
    cache = tq.alloc_cache("turbo4", n + 37, d=D2)
    tq.tq_quantize_set_rows(ctx, x_t, cache, row_ids=torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    ref, _ = Codec("turbo4", d=D2, rotation="wht", rot_seed=5).encode(x32)
    got = host_rows(cache, n + 37)
    assert np.array_equal(got[slots], ref)
    untouched = np.setdiff1d(np.arange(n + 37), slots)
    assert np.all(got[untouched] == 0)
    assert tq.tq_ctx_device_status(ctx) == 0


def test_write_dense_band_and_zero_row():
    tq = lib()
    n = 600
    x = rows(n, 3, 2.0)
    x[7] = 0.0
    x_t, x32 = torch_rows(x, "f32")
    ctx = tq.Ctx("turbo4", "dense", 6, d=D2)
    cache = tq.alloc_cache("turbo4", n, d=D2)
    tq.tq_quantize_set_rows(ctx, x_t, cache)
    codec = Codec("turbo4", d=D2, rotation="dense", rot_seed=6)
    ref, aux = codec.encode(x32)
    got = host_rows(cache, n)
    assert np.array_equal(got[:, 0:4], ref[:, 0:4]) and np.array_equal(got[:, 68:72], ref[:, 68:72])
    norms, idx = oracle.unpack_turbo4_rows(got, D2)
    ok, n_diff = band_ok(idx, aux["idx"], aux["y"], codec.b32)
    assert ok, f"{n_diff} indices differ outside the 1e-5 band"
    assert np.all(idx[7] == 7) and np.all(norms[7] == 0.0)


@pytest.mark.parametrize("rot", ["wht", "dense"])
@pytest.mark.parametrize("unrotate", [True, False])
def test_dequantize(rot, unrotate):
    import torch
    tq = lib()
    n = 300
    codec = Codec("turbo4", d=D2, rotation=rot, rot_seed=9)
    blk, _ = codec.encode(rows(n, 4, 1.5))
    cache = tq.alloc_cache("turbo4", n, d=D2)
    cache[: blk.size].copy_(torch.from_numpy(blk.reshape(-1).copy()))
    ctx = tq.Ctx("turbo4", rot, 9, d=D2)
    out = torch.empty((n, D2), dtype=torch.float32, device="cuda")
    tq.tq_dequantize(ctx, cache, n, out, unrotate=unrotate)
    ref = codec.dequantize(blk, unrotate=unrotate)
    assert np.max(np.abs(out.cpu().numpy() - ref)) < 1e-4 * max(1.0, np.abs(ref).max())


CASES = [
    # B, Hq, Hkv, L, lens
    (2, 8, 2, 300, [137, 300]),
    (1, 1, 1, 512, None),
    (3, 6, 1, 1000, [1, 999, 1000]),
    (1, 12, 2, 700, None),
    (2, 8, 8, 129, [64, 129]),
]


def upload(tq, blk):
    import torch
    t = tq.alloc_cache("turbo4", blk.shape[0], d=D2)
    t[: blk.size].copy_(torch.from_numpy(blk.reshape(-1).copy()))
    return t


@pytest.mark.parametrize("rot", ["wht", "dense"])
@pytest.mark.parametrize("case", CASES)
def test_decode_parity(rot, case):
    import torch
    tq = lib()
    B, Hq, Hkv, L, lens = case
    kc = Codec("turbo4", d=D2, rotation=rot, rot_seed=11)
    vc = Codec("turbo4", d=D2, rotation=rot, rot_seed=12)
    kb, _ = kc.encode(rows(B * Hkv * L, 13, 2.0))
    vb, _ = vc.encode(rows(B * Hkv * L, 14))
    q_t, q32 = torch_rows(np.random.default_rng(15).standard_normal((B, Hq, D2)).astype(np.float32), "bf16")
    kctx, vctx = tq.Ctx("turbo4", rot, 11, d=D2), tq.Ctx("turbo4", rot, 12, d=D2)
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    out = torch.full((B, Hq, D2), float("nan"), dtype=torch.float32, device="cuda")
    sl = None if lens is None else torch.tensor(np.asarray(lens, np.int32), device="cuda")
    tq.tq_decode_attention(kctx, vctx, q_t, upload(tq, kb), upload(tq, vb), out, ws, B, Hq, Hkv, L, seq_lens=sl)
    torch.cuda.synchronize()
    kh = kc.dequantize(kb).reshape(B, Hkv, L, D2)
    vh = vc.dequantize(vb).reshape(B, Hkv, L, D2)
    ref, _ = oracle.attention_reference(q32, kh, vh, lens)
    check_outputs(out.cpu().numpy(), ref)
    assert tq.tq_ctx_device_status(kctx) == 0


def test_decode_own_block_norms_staged_and_step():
    """Each 128-element block scales by its own stored norm (second blocks rescaled 0.5-2x,
    some zero), for keys and values; the staged calls and the decode step agree with the
    one-call decode."""
    import torch
    tq = lib()
    B, Hq, Hkv, L = 2, 8, 2, 420
    rng = np.random.default_rng(21)
    kc = Codec("turbo4", d=D2, rotation="dense", rot_seed=21)
    vc = Codec("turbo4", d=D2, rotation="wht", rot_seed=22)
    kb = kc.encode(rows(B * Hkv * L, 22, 1.5))[0].copy()
    vb = vc.encode(rows(B * Hkv * L, 23))[0].copy()
    for blk in (kb, vb):
        n = blk[:, 68:72].copy().view("<f4") * rng.uniform(0.5, 2.0, (len(blk), 1)).astype(np.float32)
        n[rng.random(len(blk)) < 0.02] = 0.0
        blk[:, 68:72] = n.view(np.uint8)
    q_t, q32 = torch_rows(rng.standard_normal((B, Hq, D2)).astype(np.float32), "f32")
    kctx, vctx = tq.Ctx("turbo4", "dense", 21, d=D2), tq.Ctx("turbo4", "wht", 22, d=D2)
    kd, vd = upload(tq, kb), upload(tq, vb)
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    outs = []
    for mode in ("one", "staged", "merge"):
        out = torch.full((B, Hq, D2), float("nan"), dtype=torch.float32, device="cuda")
        if mode == "one":
            tq.tq_decode_attention(kctx, vctx, q_t, kd, vd, out, ws, B, Hq, Hkv, L)
        elif mode == "staged":
            tq.tq_decode_prepare_q(kctx, vctx, q_t, ws, B, Hq, Hkv, L)
            tq.tq_decode_partial(kctx, vctx, kd, vd, ws, B, Hq, Hkv, L)
            tq.tq_decode_combine(kctx, vctx, out, ws, B, Hq, Hkv, L)
        else:
            tq.tq_decode_prepare_q(kctx, vctx, q_t, ws, B, Hq, Hkv, L)
            tq.tq_decode_partial_merge(kctx, vctx, kd, vd, out, ws, B, Hq, Hkv, L)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    ref, _ = oracle.attention_reference(q32, kc.dequantize(kb).reshape(B, Hkv, L, D2),
                                        vc.dequantize(vb).reshape(B, Hkv, L, D2))
    check_outputs(outs[0], ref)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    assert tq.tq_decode_num_launches(kctx, vctx, B, Hq, Hkv, L) == 3
    # one decode step: the new rows at the last slot of every unit, then the decode
    new_k, nk32 = torch_rows(rows(B * Hkv, 24), "bf16")
    new_v, nv32 = torch_rows(rows(B * Hkv, 25), "bf16")
    slots = torch.tensor([(u + 1) * L - 1 for u in range(B * Hkv)], dtype=torch.int64, device="cuda")
    out = torch.full((B, Hq, D2), float("nan"), dtype=torch.float32, device="cuda")
    tq.tq_decode_step(kctx, vctx, new_k, new_v, q_t, kd, vd, out, ws, B, Hq, Hkv, L, row_ids=slots)
    torch.cuda.synchronize()
    # the oracle's own encoding of the new rows in the oracle's caches
    sl_h = slots.cpu().numpy()
    kb2, vb2 = kb.copy(), vb.copy()
    kb2[sl_h], vb2[sl_h] = kc.encode(nk32)[0], vc.encode(nv32)[0]
    got_k = host_rows(kd, B * Hkv * L)
    assert np.array_equal(got_k[sl_h][:, :4], kb2[sl_h][:, :4]) and np.array_equal(vb2[sl_h], host_rows(vd, B * Hkv * L)[sl_h])
    ref2, _ = oracle.attention_reference(q32, kc.dequantize(kb2).reshape(B, Hkv, L, D2),
                                         vc.dequantize(vb2).reshape(B, Hkv, L, D2))
    check_outputs(out.cpu().numpy(), ref2)
    assert tq.tq_ctx_device_status(kctx) == 0 and tq.tq_ctx_device_status(vctx) == 0


def test_d256_limits():
    import torch
    tq = lib()
    k2 = tq.Ctx("turbo4", "wht", 1, d=D2)
    k1 = tq.Ctx("turbo4", "wht", 1)
    with pytest.raises(tq.TQError) as e:
        tq.Ctx("turbo3", "wht", 1, d=D2)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_workspace_size(k2, k1, 1, 4, 1, 64)  # mixed head dimensions
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    with pytest.raises(tq.TQError) as e:
        tq.tq_prefill_workspace_size(k2, k2, 1, 4, 4, 1, 64)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(k2, k2, 1, 4, 1, 64))
    q = torch.zeros((1, 4, D2), dtype=torch.float32, device="cuda")
    c = tq.alloc_cache("turbo4", 64, d=D2)
    out = torch.zeros((1, 4, D2), dtype=torch.float32, device="cuda")
    sc = torch.zeros((1, 4, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention(k2, k2, q, c, c, out, ws, 1, 4, 1, 64, scores=sc)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED


def test_full_size_gqa_d256():
    """B = 2, Hq = 32, Hkv = 8, L = 32,768 at d = 256: the cache written by the GPU write path
    (dense rotation), sampled heads against the oracle on those heads' own rows."""
    import torch
    tq = lib()
    B, Hq, Hkv, L = 2, 32, 8, 32768
    kctx, vctx = tq.Ctx("turbo4", "dense", 31, d=D2), tq.Ctx("turbo4", "dense", 32, d=D2)
    kc, vc = tq.alloc_cache("turbo4", B * Hkv * L, d=D2), tq.alloc_cache("turbo4", B * Hkv * L, d=D2)
    src = {}
    for t, (ctx, cache) in enumerate(((kctx, kc), (vctx, vc))):
        x = rows(B * Hkv * L, 40 + t)
        tq.tq_quantize_set_rows(ctx, torch_rows(x, "bf16")[0], cache)
        src[t] = torch_rows(x, "bf16")[1]
    q_t, q32 = torch_rows(np.random.default_rng(42).standard_normal((B, Hq, D2)).astype(np.float32), "bf16")
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    out = torch.empty((B, Hq, D2), dtype=torch.float32, device="cuda")
    tq.tq_decode_attention(kctx, vctx, q_t, kc, vc, out, ws, B, Hq, Hkv, L)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    kcod = Codec("turbo4", d=D2, rotation="dense", rot_seed=31)
    vcod = Codec("turbo4", d=D2, rotation="dense", rot_seed=32)
    for b, h in [(0, 0), (1, 17), (1, 31)]:
        kv = oracle.gqa_kv_head(h, Hq, Hkv)
        u = (b * Hkv + kv) * L
        kh = kcod.dequantize(kcod.encode(src[0][u:u + L])[0])[None, None]
        vh = vcod.dequantize(vcod.encode(src[1][u:u + L])[0])[None, None]
        ref, _ = oracle.attention_reference(q32[b:b + 1, h:h + 1], kh, vh)
        check_outputs(o[b:b + 1, h:h + 1], ref)
