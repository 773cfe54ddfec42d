"""The benchmark's plain fp32 CPU decode loop against the oracle (CPU only).

The loop is what the benchmark reports as its CPU baseline; it must compute the same
attention as the oracle's fp64 definition, to fp32 accuracy, on one core and on
several."""

import numpy as np
import pytest

import oracle
from oracle.formats import Codec


@pytest.fixture(scope="module")
def loop():
    from oracle import build_cpu_baseline
    f = build_cpu_baseline.load()
    if f is None:
        pytest.skip("no C compiler")
    return f


@pytest.mark.parametrize("rot,B,Hq,Hkv,L", [("dense", 2, 8, 2, 300), ("wht", 1, 6, 1, 1000), ("dense", 3, 4, 4, 17)])
@pytest.mark.parametrize("threads", [1, 4])
def test_cpu_loop_matches_oracle(loop, rot, B, Hq, Hkv, L, threads):
    rng = np.random.default_rng([B, Hq, L])
    kc, vc = Codec("turbo4", rotation=rot, rot_seed=3), Codec("turbo4", rotation=rot, rot_seed=4)
    K = (rng.standard_normal((B * Hkv * L, 128)) * 2).astype(np.float32)
    V = rng.standard_normal((B * Hkv * L, 128)).astype(np.float32)
    kb, _ = kc.encode(K)
    vb, _ = vc.encode(V)
    q = rng.standard_normal((B, Hq, 128)).astype(np.float32)
    rk = np.ascontiguousarray(kc.rot.R, np.float32)
    rv = np.ascontiguousarray(vc.rot.R, np.float32)
    out = np.zeros((B, Hq, 128), np.float32)
    scale = np.float32(1 / np.sqrt(128))
    used = loop(q.ctypes.data, kb.ctypes.data, vb.ctypes.data, B, Hq, Hkv, L, rk.ctypes.data, rv.ctypes.data,
                kc.c32.ctypes.data, vc.c32.ctypes.data, scale, out.ctypes.data, threads)
    assert used >= 1
    kh = kc.dequantize(kb).reshape(B, Hkv, L, 128)
    vh = vc.dequantize(vb).reshape(B, Hkv, L, 128)
    ref, _ = oracle.attention_reference(q, kh, vh)
    assert np.max(np.abs(out - ref)) < 1e-4
