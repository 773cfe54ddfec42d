"""The decode entry point with static scratch (tq_decode_attention_static) against the
workspace entry point tq_decode_attention, through the C ABI.

Collected last on purpose: it must also pass after every other GPU test has run in the
same process.  Two calls in a row with different shapes check that nothing carries over
from one call to the next in the shared static area."""

import numpy as np
import pytest

import synth
from gpu_util import check_outputs, lib

pytestmark = pytest.mark.gpu


# (key format, rotation, seed, QJL seed), then the same for the values
PAIRS = {
    "turbo4": (("turbo4", "dense", 21, 0), ("turbo4", "wht", 22, 0)),
    "turbo3_keys": (("turbo3", "dense", 23, 0), ("turbo4", "dense", 24, 0)),
    "prod3_vgroup2": (("prod3", "dense", 25, 1025), ("vgroup2", "wht", 0, 0)),
}


def make_ctx_pair(tq, pair="turbo4"):
    return tuple(tq.Ctx(fmt, rot, seed, qjl) for fmt, rot, seed, qjl in PAIRS[pair])


def make_case(tq, B, Hq, Hkv, L, seed, pair="turbo4"):
    import torch
    kctx, vctx = make_ctx_pair(tq, pair)
    rng = np.random.default_rng(seed)
    caches = []
    for ctx, (fmt, _, _, _) in zip((kctx, vctx), PAIRS[pair]):
        x = torch.from_numpy(synth.bf16_bits(rng.standard_normal((B * Hkv * L, 128), dtype=np.float32))
                             .view(np.int16)).view(torch.bfloat16).cuda()
        cache = tq.alloc_cache(fmt, B * Hkv * L)
        tq.tq_quantize_set_rows(ctx, x, cache)
        caches.append(cache)
    q = torch.from_numpy(rng.standard_normal((B, Hq, 128), dtype=np.float32)).cuda()
    lens = torch.tensor(rng.integers(1, L + 1, size=B).astype(np.int32), device="cuda")
    return kctx, vctx, q, caches[0], caches[1], lens


def run_both(tq, case, B, Hq, Hkv, L):
    import torch
    kctx, vctx, q, kc, vc, lens = case
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    ref = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    tq.tq_decode_attention(kctx, vctx, q, kc, vc, ref, ws, B, Hq, Hkv, L, seq_lens=lens)
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    tq.tq_decode_attention_static(kctx, vctx, q, kc, vc, out, B, Hq, Hkv, L, seq_lens=lens)
    torch.cuda.synchronize()
    assert tq.tq_ctx_device_status(kctx) == 0 and tq.tq_ctx_device_status(vctx) == 0
    return out.cpu().numpy(), ref.cpu().numpy()


@pytest.mark.parametrize("pair", list(PAIRS))
def test_static_scratch_matches_workspace_entry_twice_in_a_row(pair):
    """Each (key, value) format pair has its own workspace layout (the prod3 + vgroup2
    decode adds the QJL sketch of q); every pair is run through the static area."""
    tq = lib()
    shapes = [(4, 32, 8, 5000, 1), (2, 12, 1, 700, 2)]  # larger first, then a smaller one
    for B, Hq, Hkv, L, seed in shapes:
        needed = tq.tq_decode_workspace_size(*make_ctx_pair(tq, pair), B, Hq, Hkv, L)
        assert needed <= tq.TQ_STATIC_WORKSPACE_BYTES
        case = make_case(tq, B, Hq, Hkv, L, seed, pair)
        out, ref = run_both(tq, case, B, Hq, Hkv, L)
        check_outputs(out, ref)


@pytest.mark.parametrize("pair", list(PAIRS))
def test_static_scratch_rejects_oversized_shape(pair):
    tq = lib()
    kctx, vctx = make_ctx_pair(tq, pair)
    B, Hq, Hkv, L = 64, 64, 8, 32768
    assert tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L) > tq.TQ_STATIC_WORKSPACE_BYTES
    st = tq.lib.tq_decode_attention_static(kctx.handle, vctx.handle, None, tq.TQ_DTYPE_F32, None, None, None,
                                           B, Hq, Hkv, L, 0.0, None, None)
    assert st == tq.TQ_ERR_WORKSPACE
    assert "static area" in tq.lib.tq_last_error().decode()
