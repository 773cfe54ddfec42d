"""GPU checks of tq_decode_step: one call that appends a decode step's new K / V rows to
the compressed caches and attends over the updated caches.

The call must leave exactly the cache bytes and give the outputs that the three
separate calls give (SET_ROWS of K, SET_ROWS of V, decode attention), whichever
launch plan it takes: the one-launch front (at most 256 new rows: turbo4 / turbo3 under
the dense or the WHT rotation, or prod3 keys with vgroup2 values in any rotation) or the
separate kernels (more rows).  For the turbo
formats the outputs are also checked against the oracle's attention over the caches
the call wrote, dequantized by the oracle."""

import numpy as np
import pytest

import oracle
from gpu_util import check_outputs, lib, to_host_bytes, torch_rows
from oracle.formats import Codec

pytestmark = pytest.mark.gpu


def _ctx(tq, fmt, rot, seed):
    if fmt == "prod3":
        return tq.Ctx("prod3", rot, seed, seed + 1000)
    if fmt == "vgroup2":
        return tq.Ctx("vgroup2")
    return tq.Ctx(fmt, rot, seed)


def _codec(fmt, rot, seed):
    return Codec(fmt, rotation=rot, rot_seed=seed)


def _filled_cache(tq, ctx, fmt, n, seed):
    """A cache of n rows written by the GPU write path from seeded normal rows."""
    x, _ = torch_rows(np.random.default_rng(seed).standard_normal((n, 128)).astype(np.float32), "bf16")
    c = tq.alloc_cache(fmt, n)
    tq.tq_quantize_set_rows(ctx, x, c)
    return c


def _step_inputs(B, Hq, Hkv, L, lens, seed, src):
    """New rows [B*Hkv, 128] (row b*Hkv+h is the token at position lens[b]-1 of head h of
    sequence b), their slots in the [B][Hkv][L] caches, and the step's queries."""
    import torch
    rng = np.random.default_rng(seed)
    nk, _ = torch_rows((rng.standard_normal((B * Hkv, 128)) * 2).astype(np.float32), src)
    nv, _ = torch_rows(rng.standard_normal((B * Hkv, 128)).astype(np.float32), src)
    slots = np.array([(b * Hkv + h) * L + lens[b] - 1 for b in range(B) for h in range(Hkv)], np.int64)
    q_t, q32 = torch_rows(rng.standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    return nk, nv, torch.from_numpy(slots).cuda(), q_t, q32


STEP_CASES = [
    # k_fmt, v_fmt, rotation, source dtype, B, Hq, Hkv, L, one launch for the writes and q
    ("turbo4", "turbo4", "dense", "bf16", 4, 32, 8, 1000, True),
    ("turbo4", "turbo4", "dense", "f32", 3, 12, 2, 300, True),
    ("turbo3", "turbo4", "dense", "bf16", 2, 16, 4, 700, True),
    ("turbo3", "turbo3", "dense", "bf16", 2, 16, 4, 700, True),
    ("turbo4", "turbo3", "wht", "f32", 2, 8, 2, 300, True),
    ("turbo4", "turbo4", "dense", "bf16", 32, 64, 8, 64, True),    # 256 rows, the most the front takes
    ("turbo4", "turbo4", "dense", "bf16", 33, 64, 8, 64, False),   # 264 rows
    ("turbo4", "turbo4", "wht", "bf16", 2, 8, 2, 500, True),
    ("turbo3", "turbo3", "wht", "bf16", 5, 20, 4, 200, True),      # 20 rows: a ragged row CTA
    ("turbo4", "turbo4", "wht", "bf16", 32, 64, 8, 64, True),      # 256 rows: four row CTAs per tensor
    ("turbo4", "turbo4", "wht", "bf16", 33, 64, 8, 64, False),     # 264 rows
    ("prod3", "vgroup2", "dense", "bf16", 2, 12, 2, 400, True),
    ("prod3", "vgroup2", "wht", "f32", 3, 12, 3, 300, True),
    ("prod3", "vgroup2", "dense", "bf16", 32, 64, 8, 64, True),    # 256 rows
    ("prod3", "vgroup2", "dense", "bf16", 33, 64, 8, 64, False),   # 264 rows: the separate kernels
]


@pytest.mark.parametrize("case", STEP_CASES)
def test_decode_step_matches_separate_calls(case):
    import torch
    tq = lib()
    kf, vf, rot, src, B, Hq, Hkv, L, front = case
    n_cache = B * Hkv * L
    kctx, vctx = _ctx(tq, kf, rot, 21), _ctx(tq, vf, rot, 22)
    lens = [int(x) for x in np.random.default_rng(9).integers(1, L + 1, B)]
    nk, nv, slots, q_t, q32 = _step_inputs(B, Hq, Hkv, L, lens, 10, src)
    k0, v0 = _filled_cache(tq, kctx, kf, n_cache, 11), _filled_cache(tq, vctx, vf, n_cache, 12)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))

    n_attn = tq.tq_decode_num_launches(kctx, vctx, B, Hq, Hkv, L)
    src_dt = torch.bfloat16 if src == "bf16" else torch.float32
    assert tq.tq_decode_step_num_launches(kctx, vctx, src_dt, B * Hkv, B, Hq, Hkv, L) == \
        (n_attn if front else n_attn + 2)

    # the three separate calls
    kc_a, vc_a = k0.clone(), v0.clone()
    out_a = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    tq.tq_quantize_set_rows(kctx, nk, kc_a, row_ids=slots)
    tq.tq_quantize_set_rows(vctx, nv, vc_a, row_ids=slots)
    tq.tq_decode_attention(kctx, vctx, q_t, kc_a, vc_a, out_a, ws, B, Hq, Hkv, L, seq_lens=sl)
    # one call, twice (the per-unit counters reset in between)
    kc_b, vc_b = k0.clone(), v0.clone()
    out_b = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    for _ in range(2):
        tq.tq_decode_step(kctx, vctx, nk, nv, q_t, kc_b, vc_b, out_b, ws, B, Hq, Hkv, L, row_ids=slots,
                          seq_lens=sl)
    torch.cuda.synchronize()
    assert torch.equal(kc_a, kc_b) and torch.equal(vc_a, vc_b)
    # the same kernels on the same bytes; only the order in which a unit's splits are
    # merged may differ
    np.testing.assert_allclose(out_b.cpu().numpy(), out_a.cpu().numpy(), rtol=2e-6, atol=1e-7)
    assert tq.tq_ctx_device_status(kctx) == 0 and tq.tq_ctx_device_status(vctx) == 0
    # the new rows are there: the slots changed
    kb = to_host_bytes(kc_b, n_cache, kctx.row_bytes)
    kb0 = to_host_bytes(k0, n_cache, kctx.row_bytes)
    assert np.any(kb[slots.cpu().numpy()] != kb0[slots.cpu().numpy()])

    if kf in ("turbo4", "turbo3") and vf in ("turbo4", "turbo3"):
        vb = to_host_bytes(vc_b, n_cache, vctx.row_bytes)
        kh = _codec(kf, rot, 21).dequantize(kb).reshape(B, Hkv, L, 128)
        vh = _codec(vf, rot, 22).dequantize(vb).reshape(B, Hkv, L, 128)
        ref, _ = oracle.attention_reference(q32, kh, vh, lens)
        check_outputs(out_b.cpu().numpy(), ref)


def test_decode_step_identity_slots_and_no_rows():
    """row_ids = None writes rows 0..n-1; n_rows = 0 is a plain decode."""
    import torch
    tq = lib()
    B, Hq, Hkv, L = 1, 8, 2, 256
    kctx, vctx = _ctx(tq, "turbo4", "dense", 31), _ctx(tq, "turbo4", "dense", 32)
    k0, v0 = _filled_cache(tq, kctx, "turbo4", B * Hkv * L, 1), _filled_cache(tq, vctx, "turbo4", B * Hkv * L, 2)
    nk, nv, _, q_t, _ = _step_inputs(B, Hq, Hkv, L, [L], 3, "bf16")
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    kc_a, vc_a, kc_b, vc_b = k0.clone(), v0.clone(), k0.clone(), v0.clone()
    out_a = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    out_b = torch.empty_like(out_a)
    tq.tq_quantize_set_rows(kctx, nk, kc_a)
    tq.tq_quantize_set_rows(vctx, nv, vc_a)
    tq.tq_decode_attention(kctx, vctx, q_t, kc_a, vc_a, out_a, ws, B, Hq, Hkv, L)
    tq.tq_decode_step(kctx, vctx, nk, nv, q_t, kc_b, vc_b, out_b, ws, B, Hq, Hkv, L)
    torch.cuda.synchronize()
    assert torch.equal(kc_a, kc_b) and torch.equal(vc_a, vc_b)
    np.testing.assert_allclose(out_b.cpu().numpy(), out_a.cpu().numpy(), rtol=2e-6, atol=1e-7)

    tq.tq_decode_attention(kctx, vctx, q_t, k0, v0, out_a, ws, B, Hq, Hkv, L)
    kc_c, vc_c = k0.clone(), v0.clone()
    tq.tq_decode_step(kctx, vctx, nk[:0], nv[:0], q_t, kc_c, vc_c, out_b, ws, B, Hq, Hkv, L)
    torch.cuda.synchronize()
    assert torch.equal(kc_c, k0) and torch.equal(vc_c, v0)
    np.testing.assert_allclose(out_b.cpu().numpy(), out_a.cpu().numpy(), rtol=2e-6, atol=1e-7)
    assert tq.tq_decode_step_num_launches(kctx, vctx, torch.bfloat16, 0, B, Hq, Hkv, L) == \
        tq.tq_decode_num_launches(kctx, vctx, B, Hq, Hkv, L)


def test_decode_step_rejects_bad_arguments_before_writing():
    """A failing check launches nothing: the caches keep their bytes."""
    import torch
    tq = lib()
    B, Hq, Hkv, L = 1, 4, 1, 64
    kctx, vctx = _ctx(tq, "turbo4", "dense", 41), _ctx(tq, "turbo4", "dense", 42)
    k0, v0 = _filled_cache(tq, kctx, "turbo4", L, 1), _filled_cache(tq, vctx, "turbo4", L, 2)
    nk, nv, slots, q_t, _ = _step_inputs(B, Hq, Hkv, L, [L], 3, "bf16")
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    kc, vc = k0.clone(), v0.clone()

    def call(nk_=nk, nv_=nv, ws_=ws, Hq_=Hq, Hkv_=Hkv):
        with pytest.raises(tq.TQError) as e:
            tq.tq_decode_step(kctx, vctx, nk_, nv_, q_t, kc, vc, out, ws_, B, Hq_, Hkv_, L, row_ids=slots)
        return e.value.status

    assert call(ws_=tq.alloc_workspace(256)) == tq.TQ_ERR_WORKSPACE
    assert call(nk_=nk.half(), nv_=nv.half()) == tq.TQ_ERR_UNSUPPORTED      # fp16 rows are not a source type
    buf = torch.zeros(2 * nk.numel() + 8, dtype=nk.dtype, device="cuda")
    off_k, off_v = buf[1:1 + nk.numel()].view(nk.shape), buf[5 + nk.numel():5 + 2 * nk.numel()].view(nk.shape)
    assert call(nk_=off_k, nv_=off_v) == tq.TQ_ERR_ALIGNMENT                # rows off their 8-byte boundary
    with pytest.raises(ValueError):                                          # one source dtype for K and V
        tq.tq_decode_step(kctx, vctx, nk, nv.half(), q_t, kc, vc, out, ws, B, Hq, Hkv, L, row_ids=slots)
    assert call(Hq_=3, Hkv_=2) == tq.TQ_ERR_INVALID_ARG                     # Hq not a multiple of Hkv
    torch.cuda.synchronize()
    assert torch.equal(kc, k0) and torch.equal(vc, v0)


def test_decode_step_out_of_range_slot_is_flagged():
    """A slot outside the caches is skipped and flagged in the context's device status,
    on the one-launch front as in SET_ROWS."""
    import torch
    tq = lib()
    B, Hq, Hkv, L = 1, 8, 2, 128
    kctx, vctx = _ctx(tq, "turbo4", "dense", 51), _ctx(tq, "turbo4", "dense", 52)
    k0, v0 = _filled_cache(tq, kctx, "turbo4", B * Hkv * L, 1), _filled_cache(tq, vctx, "turbo4", B * Hkv * L, 2)
    nk, nv, _, q_t, _ = _step_inputs(B, Hq, Hkv, L, [L], 3, "bf16")
    slots = torch.tensor([5, B * Hkv * L], dtype=torch.int64, device="cuda")
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    kc, vc = k0.clone(), v0.clone()
    tq.tq_decode_step(kctx, vctx, nk, nv, q_t, kc, vc, out, ws, B, Hq, Hkv, L, row_ids=slots)
    torch.cuda.synchronize()
    assert tq.tq_ctx_device_status(kctx) != 0 and tq.tq_ctx_device_status(vctx) != 0
    assert tq.tq_ctx_device_status(kctx) == 0  # cleared by the read
    kb, kb0 = to_host_bytes(kc, B * Hkv * L, 68), to_host_bytes(k0, B * Hkv * L, 68)
    changed = np.nonzero(np.any(kb != kb0, axis=1))[0]
    assert list(changed) == [5]
    assert np.all(np.isfinite(out.cpu().numpy()))


@pytest.mark.parametrize("kf,vf,rot,src,host", [("turbo4", "turbo4", "dense", "bf16", "pinned"),
                                                 ("turbo4", "turbo4", "dense", "bf16", "pageable"),
                                                 ("turbo4", "turbo4", "dense", "bf16", "pinned_in_pageable_out"),
                                                 ("turbo4", "turbo3", "dense", "f32", "pinned"),
                                                 ("turbo4", "turbo4", "wht", "bf16", "pinned"),
                                                 ("turbo4", "turbo4", "wht", "bf16", "pageable"),
                                                 ("turbo4", "turbo4", "dense/wht", "bf16", "pinned"),
                                                 ("prod3", "vgroup2", "dense", "bf16", "pinned"),
                                                 ("prod3", "vgroup2", "dense", "bf16", "pageable")])
def test_decode_step_host_buffers_match_device_call(kf, vf, rot, src, host):
    """tq_decode_step_host (one C call with host buffers) leaves the cache bytes and gives
    the outputs of tq_decode_step on the same inputs in device memory, whether it runs in
    place (page-locked input and output: the kernels read and write host memory; with the
    one-launch front, or with the separate row writes when the key and value rotations
    differ) or through the staging area (copies in and out)."""
    import torch
    tq = lib()
    B, Hq, Hkv, L = 2, 8, 2, 300
    n_cache = B * Hkv * L
    krot, vrot = rot.split("/") if "/" in rot else (rot, rot)
    kctx, vctx = _ctx(tq, kf, krot, 41), _ctx(tq, vf, vrot, 42)
    lens = [L, 200]
    nk, nv, slots, q_t, _ = _step_inputs(B, Hq, Hkv, L, lens, 43, src)
    k0, v0 = _filled_cache(tq, kctx, kf, n_cache, 44), _filled_cache(tq, vctx, vf, n_cache, 45)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    kc_a, vc_a = k0.clone(), v0.clone()
    out_a = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    tq.tq_decode_step(kctx, vctx, nk, nv, q_t, kc_a, vc_a, out_a, ws, B, Hq, Hkv, L, row_ids=slots, seq_lens=sl)
    inputs, _ = tq.pack_step_inputs(nk, nv, q_t)
    if host == "pageable":
        inputs = torch.empty(inputs.shape, dtype=inputs.dtype).copy_(inputs)
        assert not inputs.is_pinned()
    out_h = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, pin_memory=(host == "pinned"))
    staging = tq.alloc_workspace(tq.tq_decode_step_host_staging_size(kctx, nk.dtype, nk.shape[0], q_t.dtype, B, Hq))
    kc_b, vc_b = k0.clone(), v0.clone()
    tq.tq_decode_step_host(kctx, vctx, inputs, nk.dtype, nk.shape[0], q_t.dtype, out_h, slots, kc_b, vc_b, staging,
                           ws, B, Hq, Hkv, L, seq_lens=sl)
    torch.cuda.synchronize()
    assert torch.equal(kc_a, kc_b) and torch.equal(vc_a, vc_b)
    # (the CTA that completes a unit, and with it the fused merge's summation order, can
    # differ between runs)
    np.testing.assert_allclose(out_h.numpy(), out_a.cpu().numpy(), rtol=1e-5, atol=1e-6)
    assert tq.tq_ctx_device_status(kctx) == 0
    # a staging area smaller than required is refused before anything is copied or launched
    short = staging[: staging.numel() - 256]
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_step_host(kctx, vctx, inputs, nk.dtype, nk.shape[0], q_t.dtype, out_h, slots, kc_b, vc_b,
                               short, ws, B, Hq, Hkv, L, seq_lens=sl)
    assert e.value.status == tq.TQ_ERR_WORKSPACE


@pytest.mark.parametrize("pinned", [True, False])
def test_decode_step_host_no_new_rows(pinned):
    """tq_decode_step_host with n_rows = 0: the host buffer holds q alone (read in place
    when page-locked, copied otherwise), the caches are untouched, and the output is
    tq_decode_attention's."""
    import torch
    tq = lib()
    B, Hq, Hkv, L = 2, 8, 2, 300
    kctx, vctx = _ctx(tq, "turbo4", "dense", 51), _ctx(tq, "turbo4", "dense", 52)
    k0, v0 = _filled_cache(tq, kctx, "turbo4", B * Hkv * L, 53), _filled_cache(tq, vctx, "turbo4", B * Hkv * L, 54)
    nk, nv, slots, q_t, _ = _step_inputs(B, Hq, Hkv, L, [L, 120], 55, "bf16")
    sl = torch.tensor([L, 120], dtype=torch.int32, device="cuda")
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    out_a = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    tq.tq_decode_attention(kctx, vctx, q_t, k0, v0, out_a, ws, B, Hq, Hkv, L, seq_lens=sl)
    inputs, _ = tq.pack_step_inputs(nk[:0], nv[:0], q_t)
    if not pinned:
        inputs = torch.empty(inputs.shape, dtype=inputs.dtype).copy_(inputs)
    out_h = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, pin_memory=pinned)
    staging = tq.alloc_workspace(tq.tq_decode_step_host_staging_size(kctx, nk.dtype, 0, q_t.dtype, B, Hq))
    kc, vc = k0.clone(), v0.clone()
    tq.tq_decode_step_host(kctx, vctx, inputs, nk.dtype, 0, q_t.dtype, out_h, slots, kc, vc, staging, ws,
                           B, Hq, Hkv, L, seq_lens=sl)
    torch.cuda.synchronize()
    assert torch.equal(kc, k0) and torch.equal(vc, v0)
    np.testing.assert_allclose(out_h.numpy(), out_a.cpu().numpy(), rtol=1e-5, atol=1e-6)
    assert tq.tq_ctx_device_status(kctx) == 0
