"""Every call that launches work refuses a context whose device is not the current one.

A one-GPU machine cannot make the current device differ from a context's device, so the
test records another device in the context through the testing hook
tq_test_ctx_set_device, checks that each launching call returns TQ_ERR_INVALID_ARG
without writing anything, then restores the true device and checks that the same calls
work.  Nothing is launched by the refused calls."""

import numpy as np
import pytest

from gpu_util import lib

pytestmark = pytest.mark.gpu


def test_calls_refuse_a_context_of_another_device():
    import torch
    tq = lib()
    dev = torch.cuda.current_device()
    kctx, vctx = tq.Ctx("turbo4", "dense", 31), tq.Ctx("turbo4", "wht", 32)
    B, Hq, Hkv, L = 2, 8, 2, 300
    rows = B * Hkv * L
    x = torch.randn(rows, 128, dtype=torch.float32, device="cuda")
    kc, vc = tq.alloc_cache("turbo4", rows), tq.alloc_cache("turbo4", rows)
    tq.tq_quantize_set_rows(kctx, x, kc)
    tq.tq_quantize_set_rows(vctx, x, vc)
    q = torch.randn(B, Hq, 128, dtype=torch.float32, device="cuda")
    ws = tq.alloc_workspace(tq.tq_decode_workspace_size(kctx, vctx, B, Hq, Hkv, L))
    torch.cuda.synchronize()
    kc_before = kc.clone()
    out = torch.full((B, Hq, 128), float("nan"), device="cuda")
    deq = torch.full((4, 128), float("nan"), device="cuda")

    def calls():
        s = tq.lib
        n = tq._sz(0)
        stream = torch.cuda.current_stream().cuda_stream
        return {
            "set_rows": s.tq_quantize_set_rows(kctx.handle, x.data_ptr(), tq.TQ_DTYPE_F32, 4, 128, None,
                                               kc.data_ptr(), rows, stream),
            "dequantize": s.tq_dequantize(kctx.handle, kc.data_ptr(), 4, 1, deq.data_ptr(), stream),
            "workspace_size": s.tq_decode_workspace_size(kctx.handle, vctx.handle, B, Hq, Hkv, L,
                                                         tq.ctypes.byref(n)),
            "decode": s.tq_decode_attention(kctx.handle, vctx.handle, q.data_ptr(), tq.TQ_DTYPE_F32,
                                            kc.data_ptr(), vc.data_ptr(), None, B, Hq, Hkv, L, 0.0,
                                            out.data_ptr(), None, ws.data_ptr(), ws.numel(), stream),
            "decode_static": s.tq_decode_attention_static(kctx.handle, vctx.handle, q.data_ptr(),
                                                          tq.TQ_DTYPE_F32, kc.data_ptr(), vc.data_ptr(), None,
                                                          B, Hq, Hkv, L, 0.0, out.data_ptr(), stream),
            "prefill_size": s.tq_prefill_workspace_size(kctx.handle, vctx.handle, B, 4, Hq, Hkv, L,
                                                        tq.ctypes.byref(n)),
        }

    # both contexts on another device than the current one: every call refused
    tq.lib.tq_test_ctx_set_device(kctx.handle, dev + 1)
    tq.lib.tq_test_ctx_set_device(vctx.handle, dev + 1)
    st = calls()
    assert all(v == tq.TQ_ERR_INVALID_ARG for v in st.values()), st
    torch.cuda.synchronize()
    assert torch.equal(kc, kc_before)
    assert torch.isnan(out).all() and torch.isnan(deq).all()
    # only the value context elsewhere: the calls taking both contexts are refused
    tq.lib.tq_test_ctx_set_device(kctx.handle, dev)
    st = calls()
    for name in ("workspace_size", "decode", "decode_static", "prefill_size"):
        assert st[name] == tq.TQ_ERR_INVALID_ARG, (name, st)
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    # the true device again: the same calls run
    tq.lib.tq_test_ctx_set_device(kctx.handle, dev)
    tq.lib.tq_test_ctx_set_device(vctx.handle, dev)
    st = calls()
    assert all(v == tq.TQ_OK for v in st.values()), st
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(deq).all()
    assert tq.tq_ctx_device_status(kctx) == 0
