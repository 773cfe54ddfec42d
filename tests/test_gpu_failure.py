"""Failure detection on the GPU without a fault: every wait in the decode kernel is
bounded (about 2 s).  A testing hook makes the producer withhold the first tile, so the
consumers' waits run out; the kernel must record status 3 and return, and the context
must keep working."""

import numpy as np
import pytest

from gpu_util import check_outputs, lib, torch_rows
from oracle.formats import Codec
from test_gpu_decode import oracle_cache, reference, run_decode, upload_cache

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_context_stays_usable():
    import torch
    tq = lib()
    B, Hq, Hkv, L = 1, 4, 1, 1000
    codec = Codec("turbo4", rotation="wht", rot_seed=3)
    kb, vb = oracle_cache(codec, B, Hkv, L, 51), oracle_cache(codec, B, Hkv, L, 52)
    kc, vc = upload_cache(tq, "turbo4", kb), upload_cache(tq, "turbo4", vb)
    ctx = tq.Ctx("turbo4", "wht", 3)
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(ctx, ctx, B, Hq, Hkv, L))
    st = tq.lib.tq_test_decode_wait_timeout(ctx.handle, ctx.handle, kc.data_ptr(), vc.data_ptr(), B, Hq, Hkv, L,
                                            ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == tq.TQ_OK
    torch.cuda.synchronize()
    assert tq.tq_ctx_device_status(ctx) == 3
    assert tq.tq_ctx_device_status(ctx) == 0  # cleared by the read
    # the same context decodes correctly afterwards
    q_t, q32 = torch_rows(np.random.default_rng(53).standard_normal((B, Hq, 128)).astype(np.float32), "f32")
    out, _ = run_decode(tq, ctx, ctx, q_t, kc, vc, B, Hq, Hkv, L, scores=False)
    ref, _ = reference(q32, codec, kb, codec, vb, None)
    check_outputs(out, ref)
    assert tq.tq_ctx_device_status(ctx) == 0
