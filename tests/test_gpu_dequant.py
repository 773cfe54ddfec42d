"""GPU parity of tq_dequantize (the boundary reconstruction) against the oracle.

The packed rows are encoded by the oracle, so both sides decode identical bytes.  The
GPU reconstructs in fp32 (a 128-term dot product per element when un-rotating), the
oracle in fp64: the bound is 1e-5 of the row's largest magnitude, about 100 fp32 ulps
of headroom over a 128-term sum.  Without un-rotation each element is one product (or
one multiply-add for group values), so the bound is a few ulps."""

import numpy as np
import pytest

from gpu_util import lib
from oracle.formats import Codec

pytestmark = pytest.mark.gpu

CASES = [
    ("turbo4", "wht"), ("turbo4", "dense"),
    ("turbo3", "wht"), ("turbo3", "dense"),
    ("prod3", "dense"),
    ("vgroup2", None),
]


def rows(n, seed):
    x = (np.random.default_rng(seed).standard_normal((n, 128)) * 3.0).astype(np.float32)
    x[0] = 0.0                       # zero row: norm 0
    x[1] *= 1e-3                     # small
    x[2, :64] = 5.0                  # two constant groups
    return x


def gpu_dequantize(tq, ctx, blocks, unrotate):
    import torch
    n = blocks.shape[0]
    cache = tq.alloc_cache(ctx.fmt, n)
    flat = torch.from_numpy(blocks.reshape(-1).copy())
    cache[: flat.numel()].copy_(flat)
    dst = torch.full((n, 128), float("nan"), dtype=torch.float32, device="cuda")
    tq.tq_dequantize(ctx, cache, n, dst, unrotate=unrotate)
    torch.cuda.synchronize()
    return dst.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("fmt,rot", CASES)
@pytest.mark.parametrize("unrotate", [True, False])
def test_dequantize_matches_oracle(fmt, rot, unrotate):
    tq = lib()
    x = rows(777, 31)
    if fmt == "prod3":
        codec, ctx = Codec(fmt, rotation=rot, rot_seed=3, qjl_seed=1003), tq.Ctx(fmt, rot, 3, 1003)
    elif fmt == "vgroup2":
        codec, ctx = Codec(fmt), tq.Ctx(fmt)
    else:
        codec, ctx = Codec(fmt, rotation=rot, rot_seed=8), tq.Ctx(fmt, rot, 8)
    blocks, _ = codec.encode(x)
    got = gpu_dequantize(tq, ctx, blocks, unrotate)
    ref = codec.dequantize(blocks, unrotate=unrotate)
    assert np.all(np.isfinite(got))
    scale = np.maximum(np.abs(ref).max(axis=1, keepdims=True), 1e-30)
    err = np.abs(got - ref) / scale
    one_product = (not unrotate and fmt in ("turbo4", "turbo3")) or fmt == "vgroup2"
    bound = 1e-6 if one_product else 1e-5
    assert err.max() <= bound, f"max error {err.max():.3e} of the row scale > {bound}"
    assert np.all(got[0] == 0.0)  # a zero row reconstructs to zero


@pytest.mark.parametrize("fmt,rot,kind", [("turbo4", "wht", "sphere"), ("turbo3", "dense", "sphere"),
                                          ("prod3", "dense", "sphere")])
def test_dequantize_other_codebooks_and_shrunk_qjl(fmt, rot, kind):
    """The sphere-marginal codebook for each rotated format, and the 2/pi-shrunk QJL term."""
    tq = lib()
    x = rows(500, 37)
    if fmt == "prod3":
        codec = Codec(fmt, rotation=rot, rot_seed=3, qjl_seed=1003, codebook=kind, qjl_shrink=True)
        ctx = tq.Ctx(fmt, rot, 3, 1003, codebook=kind, qjl_shrink=True)
    else:
        codec, ctx = Codec(fmt, rotation=rot, rot_seed=8, codebook=kind), tq.Ctx(fmt, rot, 8, codebook=kind)
    blocks, _ = codec.encode(x)
    got = gpu_dequantize(tq, ctx, blocks, True)
    ref = codec.dequantize(blocks, unrotate=True)
    scale = np.maximum(np.abs(ref).max(axis=1, keepdims=True), 1e-30)
    assert (np.abs(got - ref) / scale).max() <= 1e-5
