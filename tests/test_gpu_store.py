"""GPU tests of the ring-buffer capture + block-append store against the oracle.

After every append the store must hold: len tokens; flushed = the blocks the ring had to
give up (ring_tokens/2 at a time, only when full); compressed rows [0, flushed) of every
(sequence, KV head) equal to the oracle's encoding of those tokens (bit-exact under the
WHT rotation); and decode over the store equal to the oracle's attention over the
dequantized prefix followed by the exact bf16 tail."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import check_outputs, lib, torch_rows
from oracle.formats import Codec

pytestmark = pytest.mark.gpu


def tokens(B, Hkv, N, seed, scale=1.0):
    """bf16 token rows [B, Hkv, N, 128]: (exact fp32 values, bf16 bits)."""
    x = (np.random.default_rng(seed).standard_normal((B, Hkv, N, 128)) * scale).astype(np.float32)
    bits = synth.bf16_bits(x)
    return synth.bf16_to_f32(bits), bits


def to_dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def expected_flushed(n, R):
    return 0 if n <= R else -(-(n - R) // (R // 2)) * (R // 2)


def check_store(tq, st, kcod, vcod, kx, vx, n, R, q32, q_t, Hq, fmt_k="turbo4"):
    import torch
    B, Hkv = kx.shape[0], kx.shape[1]
    length, flushed, _, _ = st.state()
    assert length == n and flushed == expected_flushed(n, R)
    L = st.L
    rb = {"turbo4": 68, "turbo3": 56, "prod3": 56}[fmt_k]
    kbytes = st.cache_bytes("k").cpu().numpy()[: B * Hkv * L * rb].reshape(B, Hkv, L, rb)
    vrb = {"vgroup2": 48, "turbo3": 56}.get(vcod.fmt, 68)
    vbytes = st.cache_bytes("v").cpu().numpy()[: B * Hkv * L * vrb].reshape(B, Hkv, L, vrb)
    if flushed:
        ref_k, _ = kcod.encode(kx[:, :, :flushed].reshape(-1, 128))
        ref_v, _ = vcod.encode(vx[:, :, :flushed].reshape(-1, 128))
        assert np.array_equal(kbytes[:, :, :flushed].reshape(-1, rb), ref_k), "compressed keys differ"
        assert np.array_equal(vbytes[:, :, :flushed].reshape(-1, vrb), ref_v), "compressed values differ"
    # the oracle: dequantized prefix, then the exact tail
    kh = np.concatenate([kcod.dequantize(kbytes[:, :, :flushed].reshape(-1, rb)).reshape(B, Hkv, flushed, 128),
                         kx[:, :, flushed:n].astype(np.float64)], axis=2)
    vh = np.concatenate([vcod.dequantize(vbytes[:, :, :flushed].reshape(-1, vrb)).reshape(B, Hkv, flushed, 128),
                         vx[:, :, flushed:n].astype(np.float64)], axis=2)
    ref, _ = oracle.attention_reference(q32, kh, vh)
    ws = tq.alloc_workspace(st.workspace_size(Hq))
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    st.decode(q_t, out, ws, Hq)
    torch.cuda.synchronize()
    check_outputs(out.cpu().numpy(), ref)


def test_store_one_token_at_a_time():
    """Decode-style appends: the ring fills, then gives up half of itself every 32 tokens;
    checked while everything is still exact, just after the first flush and later."""
    tq = lib()
    B, Hkv, Hq, L, R, N = 2, 2, 8, 512, 64, 150
    kcod, vcod = Codec("turbo4", rotation="wht", rot_seed=61), Codec("turbo4", rotation="wht", rot_seed=62)
    kctx, vctx = tq.Ctx("turbo4", "wht", 61), tq.Ctx("turbo4", "wht", 62)
    kx, kb = tokens(B, Hkv, N, 61, scale=2.0)
    vx, vb = tokens(B, Hkv, N, 62)
    q_t, q32 = torch_rows(np.random.default_rng(63).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    st = tq.Store(kctx, vctx, B, Hkv, L, R)
    kd, vd = to_dev(kb), to_dev(vb)
    for t in range(N):
        st.append(kd[:, :, t:t + 1].contiguous(), vd[:, :, t:t + 1].contiguous())
        if t + 1 in (10, 65, 150):
            check_store(tq, st, kcod, vcod, kx, vx, t + 1, R, q32, q_t, Hq)
    assert tq.tq_ctx_device_status(kctx) == 0 and tq.tq_ctx_device_status(vctx) == 0


def test_store_chunked_appends_cross_several_flushes():
    """Appends larger than the ring flush several blocks inside one call; turbo3 keys."""
    tq = lib()
    B, Hkv, Hq, L, R = 1, 2, 8, 400, 32
    kcod, vcod = Codec("turbo3", rotation="wht", rot_seed=71), Codec("turbo4", rotation="wht", rot_seed=72)
    kctx, vctx = tq.Ctx("turbo3", "wht", 71), tq.Ctx("turbo4", "wht", 72)
    chunks = [37, 100, 5, 64, 1]
    N = sum(chunks)
    kx, kb = tokens(B, Hkv, N, 71, scale=2.0)
    vx, vb = tokens(B, Hkv, N, 72)
    q_t, q32 = torch_rows(np.random.default_rng(73).standard_normal((B, Hq, 128)).astype(np.float32), "f32")
    st = tq.Store(kctx, vctx, B, Hkv, L, R)
    kd, vd = to_dev(kb), to_dev(vb)
    t = 0
    for c in chunks:
        st.append(kd[:, :, t:t + c].contiguous(), vd[:, :, t:t + c].contiguous())
        t += c
        check_store(tq, st, kcod, vcod, kx, vx, t, R, q32, q_t, Hq, fmt_k="turbo3")


def test_store_symmetric_turbo3():
    """turbo3 keys and turbo3 values (the 3.5-bit cache of the post-mortem's section 1)."""
    tq = lib()
    B, Hkv, Hq, L, R = 2, 2, 8, 300, 32
    kcod, vcod = Codec("turbo3", rotation="wht", rot_seed=91), Codec("turbo3", rotation="wht", rot_seed=92)
    kctx, vctx = tq.Ctx("turbo3", "wht", 91), tq.Ctx("turbo3", "wht", 92)
    chunks = [20, 50, 3, 40]
    N = sum(chunks)
    kx, kb = tokens(B, Hkv, N, 91, scale=2.0)
    vx, vb = tokens(B, Hkv, N, 92)
    q_t, q32 = torch_rows(np.random.default_rng(93).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    st = tq.Store(kctx, vctx, B, Hkv, L, R)
    kd, vd = to_dev(kb), to_dev(vb)
    t = 0
    for c in chunks:
        st.append(kd[:, :, t:t + c].contiguous(), vd[:, :, t:t + c].contiguous())
        t += c
        check_store(tq, st, kcod, vcod, kx, vx, t, R, q32, q_t, Hq, fmt_k="turbo3")
    assert tq.tq_ctx_device_status(kctx) == 0 and tq.tq_ctx_device_status(vctx) == 0


def test_store_prod3_keys_group_values():
    """prod3 keys with vgroup2 values (values are not rotated: the exact tail is merged
    without a rotation)."""
    tq = lib()
    B, Hkv, Hq, L, R, N = 2, 1, 6, 300, 16, 70
    kcod = Codec("prod3", rotation="dense", rot_seed=81, qjl_seed=1081)
    vcod = Codec("vgroup2")
    kctx, vctx = tq.Ctx("prod3", "dense", 81, 1081), tq.Ctx("vgroup2")
    kx, kb = tokens(B, Hkv, N, 81)
    vx, vb = tokens(B, Hkv, N, 82, scale=3.0)
    q_t, q32 = torch_rows(np.random.default_rng(83).standard_normal((B, Hq, 128)).astype(np.float32), "bf16")
    st = tq.Store(kctx, vctx, B, Hkv, L, R)
    st.append(to_dev(kb), to_dev(vb))
    # dense rotation: the written keys may differ from the oracle's only in the boundary band,
    # so compare decode against the oracle's reading of the bytes the GPU wrote
    import torch
    length, flushed, _, _ = st.state()
    assert length == N and flushed == expected_flushed(N, R)
    kbytes = st.cache_bytes("k").cpu().numpy()[: B * Hkv * L * 56].reshape(B, Hkv, L, 56)
    vbytes = st.cache_bytes("v").cpu().numpy()[: B * Hkv * L * 48].reshape(B, Hkv, L, 48)
    assert np.array_equal(vbytes[:, :, :flushed].reshape(-1, 48), vcod.encode(vx[:, :, :flushed].reshape(-1, 128))[0])
    kh = np.concatenate([kcod.dequantize(kbytes[:, :, :flushed].reshape(-1, 56)).reshape(B, Hkv, flushed, 128),
                         kx[:, :, flushed:].astype(np.float64)], axis=2)
    vh = np.concatenate([vcod.dequantize(vbytes[:, :, :flushed].reshape(-1, 48)).reshape(B, Hkv, flushed, 128),
                         vx[:, :, flushed:].astype(np.float64)], axis=2)
    ref, _ = oracle.attention_reference(q32, kh, vh)
    ws = tq.alloc_workspace(st.workspace_size(Hq))
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    st.decode(q_t, out, ws, Hq)
    torch.cuda.synchronize()
    check_outputs(out.cpu().numpy(), ref)


def test_store_capacity_and_argument_errors():
    import torch
    tq = lib()
    ctx = tq.Ctx("turbo4", "wht", 0)
    with pytest.raises(tq.TQError) as e:
        tq.Store(ctx, ctx, 1, 1, 64, 3)  # odd ring
    assert e.value.status == tq.TQ_ERR_INVALID_ARG
    st = tq.Store(ctx, ctx, 1, 1, 32, 16)
    _, kb = tokens(1, 1, 64, 91)
    kd = to_dev(kb)
    with pytest.raises(tq.TQError) as e:  # 60 tokens would need 48 compressed rows > 32
        st.append(kd[:, :, :60].contiguous(), kd[:, :, :60].contiguous())
    assert e.value.status == tq.TQ_ERR_INVALID_ARG
    assert st.state()[:2] == (0, 0)  # nothing appended
    ws = tq.alloc_workspace(st.workspace_size(4))
    out = torch.empty((1, 4, 128), dtype=torch.float32, device="cuda")
    q = torch.zeros((1, 4, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TQError) as e:  # empty store
        st.decode(q, out, ws, 4)
    assert e.value.status == tq.TQ_ERR_INVALID_ARG
    st.append(kd[:, :, :48].contiguous(), kd[:, :, :48].contiguous())  # 32 compressed + 16 exact: full
    assert st.state()[:2] == (48, 32)
    with pytest.raises(tq.TQError):
        st.append(kd[:, :, :1].contiguous(), kd[:, :, :1].contiguous())
