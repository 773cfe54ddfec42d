"""GPU parity of the chunked prefill attention (tensor-core scores and PV products over
the turbo4 cache) against the oracle's causal attention.

Caches are encoded by the oracle, so both sides attend over identical packed bytes;
outputs are compared element by element (max abs 2e-3) and per row (norm-wise
relative 1e-3).  Cases span several query tiles and key tiles with ragged tails, every
q-head grouping the kernel takes (1 to 16 q-heads per KV head), sequences that start at
position 0 and sequences whose chunk ends at the last cache row, and a long cache whose
key tiles are split over every SM."""

import numpy as np
import pytest

import oracle
from gpu_util import check_outputs, lib, torch_rows
from oracle.formats import Codec
from test_gpu_decode import oracle_cache, upload_cache

pytestmark = pytest.mark.gpu


def run_prefill(tq, kctx, vctx, q_t, kc, vc, q_start, B, T, Hq, Hkv, L):
    import torch
    ws = tq.alloc_workspace(tq.tq_prefill_workspace_size(kctx, vctx, B, T, Hq, Hkv, L))
    out = torch.full((B, T, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    qs = torch.tensor(np.asarray(q_start, np.int32), device="cuda")
    tq.tq_prefill_attention(kctx, vctx, q_t, kc, vc, qs, out, ws, B, T, Hq, Hkv, L)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def reference(q32, kcodec, kb, vcodec, vb, q_start):
    B, Hkv, L, _ = kb.shape
    kh = kcodec.dequantize(kb.reshape(-1, kb.shape[-1])).reshape(B, Hkv, L, 128)
    vh = vcodec.dequantize(vb.reshape(-1, vb.shape[-1])).reshape(B, Hkv, L, 128)
    return oracle.prefill_reference(q32, kh, vh, q_start)


CASES = [
    # B, T, Hq, Hkv, L, q_start
    (1, 64, 4, 1, 300, [236]),          # 4 q-heads per KV head: 2 query tiles, ragged last key tile
    (2, 40, 8, 2, 500, [0, 460]),       # a sequence from position 0, one ending at the last row
    (1, 20, 8, 1, 257, [100]),          # 8 q-heads per KV head: 16 queries per tile
    (1, 130, 1, 1, 700, [570]),         # no grouping: 128 queries per tile, a 2-query tail
    (2, 16, 16, 1, 1000, [0, 984]),     # 16 q-heads per KV head
]


@pytest.mark.parametrize("rot", ["wht", "dense"])
@pytest.mark.parametrize("case", CASES)
def test_prefill_parity(rot, case):
    tq = lib()
    B, T, Hq, Hkv, L, q_start = case
    kcodec = Codec("turbo4", rotation=rot, rot_seed=31)
    vcodec = Codec("turbo4", rotation=rot, rot_seed=32)
    kb = oracle_cache(kcodec, B, Hkv, L, 31, scale=2.0, dist="lognormal")
    vb = oracle_cache(vcodec, B, Hkv, L, 32)
    q_t, q32 = torch_rows(np.random.default_rng(33).standard_normal((B, T, Hq, 128)).astype(np.float32), "bf16")
    kctx, vctx = tq.Ctx("turbo4", rot, 31), tq.Ctx("turbo4", rot, 32)
    out = run_prefill(tq, kctx, vctx, q_t, upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb),
                      q_start, B, T, Hq, Hkv, L)
    ref = reference(q32, kcodec, kb, vcodec, vb, q_start)
    check_outputs(out.reshape(B * T, Hq, 128), ref.reshape(B * T, Hq, 128))
    assert tq.tq_ctx_device_status(kctx) == 0


def test_prefill_long_cache_split_over_every_sm():
    """One query tile against 20,000 keys: the key tiles of the single unit are spread
    over all SMs (about a hundred partials per row to merge); f32 queries, peaked scores."""
    tq = lib()
    B, T, Hq, Hkv, L = 1, 32, 4, 1, 20_000
    q_start = [L - T]
    codec_k = Codec("turbo4", rotation="wht", rot_seed=41)
    codec_v = Codec("turbo4", rotation="wht", rot_seed=42)
    kb = oracle_cache(codec_k, B, Hkv, L, 41, scale=3.0, dist="lognormal")
    vb = oracle_cache(codec_v, B, Hkv, L, 42)
    q_t, q32 = torch_rows(np.random.default_rng(43).standard_normal((B, T, Hq, 128)).astype(np.float32) * 2.0, "f32")
    kctx, vctx = tq.Ctx("turbo4", "wht", 41), tq.Ctx("turbo4", "wht", 42)
    out = run_prefill(tq, kctx, vctx, q_t, upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb),
                      q_start, B, T, Hq, Hkv, L)
    ref = reference(q32, codec_k, kb, codec_v, vb, q_start)
    check_outputs(out.reshape(B * T, Hq, 128), ref.reshape(B * T, Hq, 128))
    assert tq.tq_ctx_device_status(kctx) == 0


def test_prefill_matches_decode_for_the_last_query():
    """The chunk's last query attends to the whole cache: the same row as the decode."""
    import torch
    tq = lib()
    B, T, Hq, Hkv, L = 2, 24, 8, 2, 400
    codec = Codec("turbo4", rotation="dense", rot_seed=5)
    kb, vb = oracle_cache(codec, B, Hkv, L, 51), oracle_cache(codec, B, Hkv, L, 52)
    q_t, q32 = torch_rows(np.random.default_rng(53).standard_normal((B, T, Hq, 128)).astype(np.float32), "bf16")
    ctx = tq.Ctx("turbo4", "dense", 5)
    kc, vc = upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb)
    out = run_prefill(tq, ctx, ctx, q_t, kc, vc, [L - T, L - T], B, T, Hq, Hkv, L)
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(ctx, ctx, B, Hq, Hkv, L))
    dout = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    tq.tq_decode_attention(ctx, ctx, q_t[:, T - 1].contiguous(), kc, vc, dout, ws, B, Hq, Hkv, L)
    torch.cuda.synchronize()
    assert np.max(np.abs(out[:, T - 1] - dout.cpu().numpy())) <= 2e-3


def test_prefill_bad_start_is_clamped_and_flagged():
    tq = lib()
    B, T, Hq, Hkv, L = 1, 8, 4, 1, 64
    codec = Codec("turbo4", rotation="wht", rot_seed=0)
    kb, vb = oracle_cache(codec, B, Hkv, L, 61), oracle_cache(codec, B, Hkv, L, 62)
    q_t, q32 = torch_rows(np.random.default_rng(63).standard_normal((B, T, Hq, 128)).astype(np.float32), "bf16")
    ctx = tq.Ctx("turbo4", "wht", 0)
    out = run_prefill(tq, ctx, ctx, q_t, upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb),
                      [L], B, T, Hq, Hkv, L)  # past the end: clamped to L - T
    assert tq.tq_ctx_device_status(ctx) == 2
    check_outputs(out.reshape(T, Hq, 128), reference(q32, codec, kb, codec, vb, [L - T]).reshape(T, Hq, 128))


def test_prefill_rejects_bad_arguments():
    import torch
    tq = lib()
    t4, t3 = tq.Ctx("turbo4", "wht", 0), tq.Ctx("turbo3", "wht", 0)
    with pytest.raises(tq.TQError) as e:
        tq.tq_prefill_workspace_size(t3, t4, 1, 8, 4, 1, 64)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    with pytest.raises(tq.TQError) as e:
        tq.tq_prefill_workspace_size(t4, t4, 1, 8, 6, 1, 64)  # 6 q-heads per KV head
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    with pytest.raises(tq.TQError) as e:
        tq.tq_prefill_workspace_size(t4, t4, 1, 65, 4, 1, 64)  # chunk longer than the cache
    assert e.value.status == tq.TQ_ERR_INVALID_ARG
    ws = tq.alloc_workspace(256)
    q = torch.zeros((1, 8, 4, 128), dtype=torch.float32, device="cuda")
    cache = tq.alloc_cache("turbo4", 64)
    out = torch.zeros((1, 8, 4, 128), dtype=torch.float32, device="cuda")
    qs = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.tq_prefill_attention(t4, t4, q, cache, cache, qs, out, ws, 1, 8, 4, 1, 64)
    assert e.value.status == tq.TQ_ERR_WORKSPACE
