"""GPU parity of the write path (quantize / SET_ROWS) against the oracle encoder.

WHT rotation and value group quantization: packed rows bit-exact.  Dense rotation:
norm bytes bit-exact; indices may differ only within 1e-5 of a decision boundary;
prod3 residual norms within 1e-5 relative and QJL signs only where the oracle
projection is within 1e-4 of zero (rows whose indices all match)."""

import numpy as np
import pytest

import synth
from gpu_util import band_ok, lib, rows_equal_nan_aware, to_host_bytes, torch_rows
from oracle.formats import Codec, unpack_prod, unpack_turbo3, unpack_turbo4

pytestmark = pytest.mark.gpu


def special_rows():
    x = np.random.default_rng(77).standard_normal((8, 128)).astype(np.float32)
    x[0] = 0.0                      # zero vector: norm 0, every index K/2 - 1
    x[1, 3] = np.nan                # NaN propagates into the norm
    x[2] *= 1e-20                   # tiny
    x[3] *= 1e18                    # huge (squares overflow to inf)
    x[4, :] = 1.0                   # constant
    x[5, 17] = np.inf
    x[6] = -x[6]
    return x


def make_rows(n, seed, scale=1.0):
    x = (np.random.default_rng(seed).standard_normal((n, 128)) * scale).astype(np.float32)
    return np.concatenate([special_rows(), x])


def write_gpu(tq, ctx, x_t, n_rows, row_ids=None, capacity=None):
    import torch
    capacity = n_rows if capacity is None else capacity
    cache = tq.alloc_cache(ctx.fmt, capacity + 2)
    cache.fill_(0xA5)  # canary pattern everywhere, including past the last slot
    rid = None if row_ids is None else torch.from_numpy(row_ids).cuda()
    tq.tq_quantize_set_rows(ctx, x_t, cache, row_ids=rid, n_rows=n_rows)
    torch.cuda.synchronize()
    return cache


@pytest.mark.parametrize("fmt", ["turbo4", "turbo3"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("seed", [0, 5])
def test_write_wht_bit_exact(fmt, dtype, seed):
    tq = lib()
    x_t, x32 = torch_rows(make_rows(1000, seed, scale=3.0), dtype)
    ref, _ = Codec(fmt, rotation="wht", rot_seed=seed).encode(x32)
    ctx = tq.Ctx(fmt, "wht", seed)
    cache = write_gpu(tq, ctx, x_t, len(x32))
    got = to_host_bytes(cache, len(x32), ctx.row_bytes)
    bad = rows_equal_nan_aware(got, ref, fmt)
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:5]}"
    assert tq.tq_ctx_device_status(ctx) == 0


@pytest.mark.parametrize("fmt", ["turbo4", "turbo3"])
# one CTA per row / staged matrices / tensor cores; the last with several tiles per CTA
# (the row-tile ring and both accumulators reused) and a ragged last tile
@pytest.mark.parametrize("n", [100, 1000, 3000, 116786])
def test_write_dense_band(fmt, n):
    tq = lib()
    x_t, x32 = torch_rows(make_rows(n, 9, scale=2.0)[8:], "bf16")  # finite rows
    codec = Codec(fmt, rotation="dense", rot_seed=2)
    ref, aux = codec.encode(x32)
    ctx = tq.Ctx(fmt, "dense", 2)
    got = to_host_bytes(write_gpu(tq, ctx, x_t, len(x32)), len(x32), ctx.row_bytes)
    if fmt == "turbo4":
        n, idx = unpack_turbo4(got)
        assert np.array_equal(got[:, :4], ref[:, :4])
    else:
        norms, idx = unpack_turbo3(got)
        assert np.array_equal(norms, unpack_turbo3(ref)[0])
    ok, ndiff = band_ok(idx, aux["idx"], aux["y"], codec.b32)
    assert ok, f"{ndiff} indices differ outside the boundary band"


def extreme_rows():
    """Rows at the edges of the fp32 range: squares that underflow, elements whose
    quotient by the norm is tiny or subnormal, a norm that overflows."""
    g = np.random.default_rng(79).standard_normal((7, 128)).astype(np.float32)
    x = np.empty_like(g)
    x[0] = g[0] * 1e-19                         # squares partly subnormal, normal norm
    x[1] = g[1] * 1e-31                         # elements below 2^-100 ...
    x[1, 0] = 1e-18                             # ... beside one that sets the norm
    x[2] = g[2] * 1e-20                         # quotients subnormal ...
    x[2, 9] = 1e19                              # ... under a huge element
    x[3] = g[3] * 1e-25                         # every square underflows: norm 0
    x[4] = g[4] * 1e-41                         # subnormal elements
    x[5] = g[5] * 3e18                          # the sum of squares overflows: norm inf
    x[6] = g[6] * 1e-12
    x[6, ::7] = 0.0                             # exact zeros among normal elements
    return x


@pytest.mark.parametrize("fmt", ["turbo4", "turbo3"])
@pytest.mark.parametrize("rot,n", [("wht", 1000), ("dense", 100), ("dense", 1000), ("dense", 2500)])
def test_write_extreme_magnitudes(fmt, rot, n):
    """Extreme rows spread through a block of ordinary rows (n rows in all, so each dense
    kernel -- one CTA per row, staged matrices, tensor cores -- meets them): WHT rows
    bit-exact, dense rows norm-exact with indices in the boundary band."""
    tq = lib()
    x = (np.random.default_rng(80 + n).standard_normal((n, 128)) * 2.0).astype(np.float32)
    ext = extreme_rows()
    at = np.linspace(0, n - 1, len(ext)).astype(int)
    x[at] = ext
    x_t, x32 = torch_rows(x, "bf16")
    codec = Codec(fmt, rotation=rot, rot_seed=4)
    ref, aux = codec.encode(x32)
    ctx = tq.Ctx(fmt, rot, 4)
    got = to_host_bytes(write_gpu(tq, ctx, x_t, n), n, ctx.row_bytes)
    assert tq.tq_ctx_device_status(ctx) == 0
    if rot == "wht":
        bad = rows_equal_nan_aware(got, ref, fmt)
        assert bad.size == 0, f"{bad.size} rows differ, first {bad[:5]}"
        return
    if fmt == "turbo4":
        idx = unpack_turbo4(got)[1]
        assert np.array_equal(got[:, :4], ref[:, :4])
    else:
        norms, idx = unpack_turbo3(got)
        assert np.array_equal(norms, unpack_turbo3(ref)[0])
    ok, ndiff = band_ok(idx, aux["idx"], aux["y"], codec.b32)
    assert ok, f"{ndiff} indices differ outside the boundary band (rows {at})"


@pytest.mark.parametrize("n", [100, 3000])
def test_write_prod3_band(n):
    tq = lib()
    x_t, x32 = torch_rows(make_rows(n, 11, scale=2.0)[8:], "bf16")
    codec = Codec("prod3", rotation="dense", rot_seed=3, qjl_seed=1003)
    ref, aux = codec.encode(x32)
    ctx = tq.Ctx("prod3", "dense", 3, 1003)
    got = to_host_bytes(write_gpu(tq, ctx, x_t, len(x32)), len(x32), 56)
    n, gamma, idx, sb = unpack_prod(got)
    assert np.array_equal(got[:, :4], ref[:, :4])
    ok, _ = band_ok(idx, aux["idx"], aux["y"], codec.b32)
    assert ok
    same = np.all(idx == aux["idx"], axis=1)
    assert same.mean() > 0.95
    rel = np.abs(gamma[same] - aux["gamma"][same]) / aux["gamma"][same]
    assert rel.max() < 1e-5
    flip = (sb != aux["sign_bits"]) & same[:, None]
    assert np.all(np.abs(aux["z"][flip]) < 1e-4)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_write_vgroup_bit_exact(dtype):
    tq = lib()
    x = make_rows(1000, 13, scale=5.0)
    x[8, :32] = -0.0
    x[9, 32:64] = 7.0
    x_t, x32 = torch_rows(x, dtype)
    ref, _ = Codec("vgroup2").encode(x32)
    ctx = tq.Ctx("vgroup2")
    got = to_host_bytes(write_gpu(tq, ctx, x_t, len(x32)), len(x32), 48)
    bad = np.nonzero(np.any(got != ref, axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:5]}"


def test_scatter_row_ids_canaries_and_oob_flag():
    """SET_ROWS writes row i to slot row_ids[i]; slots never written keep their canary
    bytes; an out-of-range slot is skipped and flagged (status 1)."""
    import torch
    tq = lib()
    n, cap = 200, 300
    x_t, x32 = torch_rows(make_rows(n - 8, 17), "bf16")
    slots = synth.row_permutation(cap, 3)[:n].copy()
    slots[5] = cap + 10  # out of range
    ctx = tq.Ctx("turbo4", "wht", 0)
    cache = write_gpu(tq, ctx, x_t, n, row_ids=slots, capacity=cap)
    assert tq.tq_ctx_device_status(ctx) == 1
    assert tq.tq_ctx_device_status(ctx) == 0  # cleared by the read
    ref, _ = Codec("turbo4", rotation="wht", rot_seed=0).encode(x32)
    host = cache.cpu().numpy()
    rows = host[: cap * 68].reshape(cap, 68)
    live = [i for i in range(n) if i != 5]
    assert rows_equal_nan_aware(rows[slots[live]], ref[live], "turbo4").size == 0
    untouched = sorted(set(range(cap)) - set(int(s) for s in slots if s < cap))
    assert np.all(rows[untouched] == 0xA5)
    assert np.all(host[cap * 68:] == 0xA5)  # nothing written past the last slot


def test_strided_source_rows():
    """Rows taken from a wider tensor (stride > 128) quantize like contiguous rows."""
    import torch
    tq = lib()
    x = make_rows(300, 19)[8:]
    wide = np.zeros((len(x), 256), np.float32)
    wide[:, 64:192] = x
    t = torch.from_numpy(wide).cuda()[:, 64:192]
    ctx = tq.Ctx("turbo4", "wht", 1)
    cache = write_gpu(tq, ctx, t, len(x))
    ref, _ = Codec("turbo4", rotation="wht", rot_seed=1).encode(x)
    assert np.array_equal(to_host_bytes(cache, len(x), 68), ref)


def test_zero_rows_is_noop_and_bad_alignment_rejected():
    import torch
    tq = lib()
    ctx = tq.Ctx("turbo4", "wht", 0)
    cache = tq.alloc_cache("turbo4", 4)
    x = torch.zeros((4, 128), dtype=torch.float32, device="cuda")
    tq.tq_quantize_set_rows(ctx, x, cache, n_rows=0)
    raw = torch.zeros(4 * 128 + 1, dtype=torch.float32, device="cuda")
    st = tq.lib.tq_quantize_set_rows(ctx.handle, raw.data_ptr() + 4, tq.TQ_DTYPE_F32, 4, 128, None,
                                     cache.data_ptr(), 4, None)
    assert st == tq.TQ_ERR_ALIGNMENT


@pytest.mark.parametrize("fmt,rot", [("turbo4", "wht"), ("turbo3", "wht"), ("turbo4", "dense"), ("turbo3", "dense")])
def test_write_chunk_full_size(fmt, rot):
    """The 16,384-token x 8-KV-head bf16 chunk (K and V), every row checked."""
    tq = lib()
    cfg = synth.WORKLOADS["write_chunk"]
    ctx = tq.Ctx(fmt, rot, 4)
    codec = Codec(fmt, rotation=rot, rot_seed=4)
    for tensor in ("K", "V"):
        x32, bits = synth.write_rows(cfg, tensor)
        import torch
        x_t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
        got = to_host_bytes(write_gpu(tq, ctx, x_t, len(x32)), len(x32), ctx.row_bytes)
        ref, aux = codec.encode(x32)
        if rot == "wht":
            assert np.array_equal(got, ref)
        else:
            idx = unpack_turbo4(got)[1] if fmt == "turbo4" else unpack_turbo3(got)[1]
            ok, ndiff = band_ok(idx, aux["idx"], aux["y"], codec.b32)
            assert ok, f"{ndiff} indices outside the band"
    assert tq.tq_ctx_device_status(ctx) == 0


@pytest.mark.parametrize("fmt", ["turbo4", "turbo3"])
def test_write_dense_tensor_core_scatter_and_stride(fmt):
    """Batches of 2048+ bf16 rows take the tensor-core write: rows read through a tensor
    map from a wider tensor (stride 192 elements), scattered to permuted slots; an
    out-of-range slot is skipped and flagged."""
    import torch
    tq = lib()
    n, cap = 2300, 2600
    x = make_rows(n, 23, scale=2.0)[8:]
    wide = np.zeros((len(x), 192), np.float32)
    wide[:, 32:160] = x
    bits = synth.bf16_bits(wide)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()[:, 32:160]
    x32 = synth.bf16_to_f32(bits)[:, 32:160]
    slots = synth.row_permutation(cap, 5)[:len(x)].copy()
    slots[17] = cap + 3
    ctx = tq.Ctx(fmt, "dense", 6)
    cache = write_gpu(tq, ctx, t, len(x), row_ids=slots, capacity=cap)
    assert tq.tq_ctx_device_status(ctx) == 1
    codec = Codec(fmt, rotation="dense", rot_seed=6)
    ref, aux = codec.encode(x32)
    rb = ctx.row_bytes
    host = cache.cpu().numpy()
    rows = host[: cap * rb].reshape(cap, rb)
    live = np.array([i for i in range(len(x)) if i != 17])
    got = rows[slots[live]]
    if fmt == "turbo4":
        assert np.array_equal(got[:, :4], ref[live, :4])
        idx = unpack_turbo4(got)[1]
    else:
        assert np.array_equal(unpack_turbo3(got)[0], unpack_turbo3(ref[live])[0])
        idx = unpack_turbo3(got)[1]
    ok, ndiff = band_ok(idx, aux["idx"][live], aux["y"][live], codec.b32)
    assert ok, f"{ndiff} indices differ outside the boundary band"
    untouched = sorted(set(range(cap)) - set(int(s) for s in slots if s < cap))
    assert np.all(rows[untouched] == 0xA5)


@pytest.mark.parametrize("fmt", ["turbo4", "turbo3"])
def test_write_dense_tensor_core_scatter_many_tiles(fmt):
    """The tensor-core write with several tiles per CTA (the row-tile ring and the
    accumulators reused), a ragged last tile and every record scattered to a permuted
    slot: each record lands whole in its slot (norm exact, indices in the band), one
    out-of-range slot is skipped and flagged, and no other slot is touched."""
    tq = lib()
    n, cap = 40_000 + 77, 41_000
    x = make_rows(n + 8, 31, scale=2.0)[8:]
    x_t, x32 = torch_rows(x, "bf16")
    slots = synth.row_permutation(cap, 7)[:n].copy()
    slots[12_345] = -1
    ctx = tq.Ctx(fmt, "dense", 8)
    cache = write_gpu(tq, ctx, x_t, n, row_ids=slots, capacity=cap)
    assert tq.tq_ctx_device_status(ctx) == 1
    codec = Codec(fmt, rotation="dense", rot_seed=8)
    ref, aux = codec.encode(x32)
    rb = ctx.row_bytes
    rows = cache.cpu().numpy()[: cap * rb].reshape(cap, rb)
    live = np.array([i for i in range(n) if i != 12_345])
    got = rows[slots[live]]
    if fmt == "turbo4":
        assert np.array_equal(got[:, :4], ref[live, :4])
        idx = unpack_turbo4(got)[1]
    else:
        assert np.array_equal(unpack_turbo3(got)[0], unpack_turbo3(ref[live])[0])
        idx = unpack_turbo3(got)[1]
    ok, ndiff = band_ok(idx, aux["idx"][live], aux["y"][live], codec.b32)
    assert ok, f"{ndiff} indices differ outside the boundary band"
    untouched = sorted(set(range(cap)) - set(int(v) for v in slots[live]))
    assert np.all(rows[untouched] == 0xA5)


@pytest.mark.parametrize("fmt", ["turbo4", "turbo3"])
def test_write_wht_sphere_codebook_bit_exact(fmt):
    """The sphere-marginal codebook (its own boundaries and grid table) under the WHT path."""
    tq = lib()
    x_t, x32 = torch_rows(make_rows(1500, 23, scale=2.0), "bf16")
    ref, _ = Codec(fmt, rotation="wht", rot_seed=23, codebook="sphere").encode(x32)
    ctx = tq.Ctx(fmt, "wht", 23, codebook="sphere")
    got = to_host_bytes(write_gpu(tq, ctx, x_t, len(x32)), len(x32), ctx.row_bytes)
    bad = rows_equal_nan_aware(got, ref, fmt)
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:5]}"
