"""Pins of the oracle's encoders, block layouts and dequantizers."""

import math

import numpy as np
import pytest

import oracle
import synth
from oracle.formats import Codec, Rotation, nearest_index, normalize_fp32

D = 128


def rows(n, seed=0, scale=1.0):
    return (np.random.default_rng(seed).standard_normal((n, D)) * scale).astype(np.float32)


def test_block_sizes_match_pages(page_numbers):
    assert oracle.ROW_BYTES["turbo4"] == page_numbers["turbo4_block_bytes"]
    assert 68 * 8 / 128 == page_numbers["turbo4_bits_per_value"]
    assert round(256 / 68, 2) == page_numbers["turbo4_compression_vs_fp16"]
    assert (14 * 8) / 32 == page_numbers["turbo3_bits_per_value"]  # one 14-byte turbo3 block per 32 values
    assert oracle.ROW_BYTES["turbo3"] == 4 * 14


def test_turbo4_layout_by_hand():
    """Element j sits in bits 4*(j%2) of byte 4 + j/2, after a little-endian fp32 norm."""
    idx = (np.arange(D) % 16).astype(np.uint8)[None, :]
    blk = oracle.pack_turbo4(np.array([2.0], np.float32), idx)
    assert list(blk[0, :4]) == [0, 0, 0, 0x40]  # 2.0f = 0x40000000
    assert blk[0, 4] == 0x10 and blk[0, 5] == 0x32 and blk[0, 11] == 0xFE
    n, back = oracle.unpack_turbo4(blk)
    assert n[0] == 2.0 and np.array_equal(back, idx)


def test_turbo3_layout_by_hand():
    """qs[j/4] bits 2*(j%4) hold idx & 3; signs[j/8] bit j%8 holds idx >> 2; fp16 norm first."""
    idx = (np.arange(D) % 8).astype(np.uint8)[None, :]
    blk = oracle.pack_turbo3(np.array([1.0], np.float32), idx)
    for c in range(4):
        b = blk[0, 14 * c:14 * c + 14]
        assert list(b[:2]) == [0x00, 0x3C]  # fp16 1.0
        # elements 0..3 = 0,1,2,3 -> 0b11100100; elements 4..7 = 4..7 -> low bits 0,1,2,3 again
        assert b[2] == 0xE4 and b[3] == 0xE4
        # high bits: elements 4..7 of each group of 8 are set -> 0xF0
        assert list(b[10:14]) == [0xF0] * 4
    norms, back = oracle.unpack_turbo3(blk)
    assert np.all(norms == 1.0) and np.array_equal(back, idx)


@pytest.mark.parametrize("fmt", ["turbo4", "turbo3", "prod3", "vgroup2"])
def test_pack_unpack_roundtrip(fmt):
    codec = Codec(fmt, rotation="dense", rot_seed=7, qjl_seed=8)
    x = rows(64, seed=1, scale=3.0)
    blk, aux = codec.encode(x)
    assert blk.shape == (64, oracle.ROW_BYTES[fmt])
    if fmt == "turbo4":
        n, idx = oracle.unpack_turbo4(blk)
        assert np.array_equal(n, aux["n"]) and np.array_equal(idx, aux["idx"])
    elif fmt == "turbo3":
        norms, idx = oracle.unpack_turbo3(blk)
        assert np.array_equal(idx, aux["idx"])
        assert np.array_equal(norms[:, 0], aux["n"].astype(np.float16).astype(np.float32))
    elif fmt == "prod3":
        n, g, idx, sb = oracle.unpack_prod(blk)
        assert np.array_equal(n, aux["n"]) and np.array_equal(g, aux["gamma"])
        assert np.array_equal(idx, aux["idx"]) and np.array_equal(sb, aux["sign_bits"])
    else:
        codes, s, z = oracle.unpack_vgroup(blk)
        assert np.array_equal(codes, aux["codes"])
        assert np.array_equal(s, aux["scale"].astype(np.float32))


def test_turbo4_block_is_not_turbo3_layout():
    """Regression for section 2 bug 1: a turbo4 block read with the turbo3 layout is garbage."""
    codec = Codec("turbo4", rotation="wht", rot_seed=0)
    blk, aux = codec.encode(rows(16, seed=2))
    fake = np.concatenate([blk[:, 4:60], blk[:, :0]], axis=1)
    _, idx3 = oracle.unpack_turbo3(fake)
    assert not np.array_equal(idx3 & 7, aux["idx"] & 7)


def test_canonical_norm_close_to_fp64_and_tree_independent_of_lane_order():
    x = rows(1000, seed=3, scale=5.0)
    n = oracle.canonical_norm_fp32(x)
    ref = np.linalg.norm(x.astype(np.float64), axis=1)
    assert np.max(np.abs(n - ref) / ref) < 4e-7
    # every lane finishes the butterfly with the same value (commutative adds)
    sq = x * x
    p = (sq[:, 0::4] + sq[:, 1::4]) + (sq[:, 2::4] + sq[:, 3::4])
    lanes = np.arange(32)
    for h in (16, 8, 4, 2, 1):
        p = p + p[:, lanes ^ h]
    assert np.all(p == p[:, :1])


def test_zero_and_nonfinite_rows():
    codec = Codec("turbo4", rotation="wht", rot_seed=0)
    x = np.zeros((3, D), np.float32)
    x[1, 5] = np.nan
    x[2, :] = 1.0
    x[2, 7] = np.inf
    blk, aux = codec.encode(x)
    assert aux["n"][0] == 0.0 and np.all(aux["idx"][0] == 7)  # K/2 - 1: code of coordinate 0
    assert np.isnan(aux["n"][1]) and np.all(aux["idx"][1] == 0)  # NaN compares false
    assert np.isinf(aux["n"][2])
    assert np.all(codec.dequantize(blk[:1]) == 0.0)


@pytest.mark.parametrize("fmt,bits", [("turbo4", 4), ("turbo3", 3)])
@pytest.mark.parametrize("rotation", ["wht", "dense"])
def test_encode_is_nearest_centroid_of_rotated_unit_vector(fmt, bits, rotation):
    codec = Codec(fmt, rotation=rotation, rot_seed=11)
    x = rows(500, seed=4, scale=2.0)
    _, aux = codec.encode(x)
    u = x.astype(np.float64) / np.linalg.norm(x.astype(np.float64), axis=1, keepdims=True)
    y = codec.rot.forward(u)
    assert np.max(np.abs(y - aux["y"])) < 2e-6
    c = codec.c32.astype(np.float64)
    brute = np.argmin(np.abs(aux["y"][..., None] - c), axis=-1)
    assert np.array_equal(brute, aux["idx"])
    assert np.array_equal(aux["idx"], nearest_index(aux["y"], codec.b32))


@pytest.mark.parametrize("fmt,expect", [("turbo4", 0.0203), ("turbo3", 0.0345)])
def test_reconstruction_error_matches_codebook_mse(fmt, expect):
    """E||x - x_hat||^2 / ||x||^2 = d * per-coordinate MSE of the codebook (rotation makes
    each coordinate ~N(0, 1/d))."""
    codec = Codec(fmt, rotation="dense", rot_seed=5)
    x = rows(4000, seed=6, scale=1.7)
    blk, _ = codec.encode(x)
    xh = codec.dequantize(blk)
    rel = np.sum((xh - x) ** 2, axis=1) / np.sum(x.astype(np.float64) ** 2, axis=1)
    assert abs(rel.mean() - expect) / expect < 0.05


def test_dequantize_rotated_basis():
    codec = Codec("turbo4", rotation="wht", rot_seed=0)
    blk, aux = codec.encode(rows(8, seed=7))
    yr = codec.dequantize(blk, unrotate=False)
    assert np.array_equal(yr, codec.c32.astype(np.float64)[aux["idx"]] * aux["n"][:, None].astype(np.float64))
    assert np.allclose(codec.rot.inverse(yr), codec.dequantize(blk), atol=1e-12)


def test_prod_residual_in_unrotated_space_and_gamma():
    """Section 2 bug 6: the residual lives in the normalised, unrotated space."""
    codec = Codec("prod3", rotation="dense", rot_seed=3, qjl_seed=1003)
    x = rows(200, seed=8, scale=4.0)
    _, aux = codec.encode(x)
    u = normalize_fp32(x, aux["n"]).astype(np.float64)
    x_tilde = codec.rot.inverse(codec.c32.astype(np.float64)[aux["idx"]])
    assert np.allclose(np.linalg.norm(u - x_tilde, axis=1), aux["gamma"], rtol=1e-6)
    assert np.array_equal(aux["sign_bits"], (aux["z"] >= 0).astype(np.uint8))
    assert np.allclose(aux["z"], (u - x_tilde) @ codec.S32.astype(np.float64).T, atol=1e-9)


def test_prod_needs_independent_seed():
    with pytest.raises(ValueError):
        Codec("prod3", rotation="dense", rot_seed=3, qjl_seed=3)


@pytest.mark.slow
def test_qjl_inner_product_unbiased_monte_carlo():
    """E[<x_hat, y>] = <x, y> over 10^5 independent Gaussian S (paper Theorem 2), within 3 SE."""
    rng = np.random.default_rng(21)
    codec = Codec("prod3", rotation="dense", rot_seed=3, qjl_seed=1003)
    x = rng.standard_normal((1, D)).astype(np.float32)
    y = rng.standard_normal(D)
    n, gamma, idx, _, _, _ = oracle.encode_prod(x, codec.rot, codec.c32, codec.b32, codec.S32)
    u = normalize_fp32(x, n).astype(np.float64)[0]
    x_tilde = codec.rot.inverse(codec.c32.astype(np.float64)[idx])[0]
    r = u - x_tilde
    draws, chunk = 100_000, 2_000
    vals = []
    for start in range(0, draws, chunk):
        S = rng.standard_normal((chunk, D, D))
        bits, _ = oracle.qjl_sign_bits(S, np.broadcast_to(r, (chunk, D)))
        est = x_tilde[None, :] + oracle.qjl_residual_estimate(S, bits, np.full(chunk, gamma[0], np.float64))
        vals.append(float(n[0]) * (est @ y))
    vals = np.concatenate(vals)
    truth = float(x[0].astype(np.float64) @ y)
    se = vals.std(ddof=1) / math.sqrt(draws)
    assert abs(vals.mean() - truth) < 3 * se
    # and the estimator is not trivially exact: the MSE-only part alone is biased
    mse_only = float(n[0]) * (x_tilde @ y)
    assert abs(mse_only - truth) > 3 * se


def test_qjl_zero_residual_adds_nothing():
    S = np.random.default_rng(0).standard_normal((D, D))
    bits = np.ones(D, np.uint8)
    assert np.all(oracle.qjl_residual_estimate(S, bits, 0.0) == 0.0)


def test_vgroup_codes_and_bounds():
    x = rows(300, seed=9, scale=2.0)
    codes, s16, z16 = oracle.encode_vgroup(x)
    assert codes.max() <= 3
    blk = oracle.pack_vgroup(codes, s16, z16)
    codec = Codec("vgroup2")
    xh = codec.dequantize(blk)
    s = np.repeat(s16.astype(np.float64), 32, axis=1)
    # each value is within half a step of its reconstruction, up to fp16 rounding of scale/zero
    err = np.abs(xh - x)
    assert np.all(err <= 0.5 * s + 2e-3 * np.abs(x).max())
    g = x.reshape(-1, 4, 32)
    assert np.all(codes.reshape(-1, 4, 32)[np.arange(len(g))[:, None], np.arange(4)[None, :], g.argmin(2)] == 0)
    assert np.all(codes.reshape(-1, 4, 32)[np.arange(len(g))[:, None], np.arange(4)[None, :], g.argmax(2)] == 3)


def test_vgroup_layout_by_hand():
    codes = (np.arange(D) % 4).astype(np.uint8)[None, :]
    s16 = np.array([[1.0, 2.0, 0.5, 0.0]], np.float16)
    z16 = np.array([[-1.0, 0.0, 1.0, -2.0]], np.float16)
    blk = oracle.pack_vgroup(codes, s16, z16)
    assert np.all(blk[0, :32] == 0xE4)
    assert list(blk[0, 32:36]) == [0x00, 0x3C, 0x00, 0xBC]  # scale 1.0, zero -1.0
    back = Codec("vgroup2").dequantize(blk)[0]
    assert back[0] == -1.0 and back[3] == 2.0 and back[32 + 1] == 2.0 and back[127] == -2.0


def test_vgroup_constant_and_signed_zero_groups():
    x = np.zeros((2, D), np.float32)
    x[1, :32] = -0.0
    x[1, 32:64] = 5.0
    codes, s16, z16 = oracle.encode_vgroup(x)
    assert np.all(codes == 0)
    assert np.all(s16 == 0) and np.all(z16.view(np.uint16)[:, :2] != 0x8000)  # -0 folded to +0
    assert z16[1, 1] == 5.0


def test_synth_bf16_rounding():
    x = np.array([1.0, 1.00390625, 1.005859375, -3.0e38, np.inf], np.float32)
    b = synth.bf16_bits(x)
    assert list(b) == [0x3F80, 0x3F80, 0x3F81, 0xFF62, 0x7F80]
    assert np.array_equal(synth.bf16_to_f32(b)[:2], [1.0, 1.0])


def test_qjl_estimator_energy_and_shrinkage_mse():
    """For a d x d N(0,1) sketch, r_hat = sqrt(pi/2)/d |r| S^T sign(S r) has
    E |r_hat|^2 = (pi/2 + (d-1)/d) |r|^2 (diagonal terms d^2, off-diagonal d(d-1) 2/pi),
    so scaling it by s gives MSE(s) = s^2 kappa - 2 s + 1 (units of |r|^2).  Monte Carlo over
    independent sketches pins both, including the 2/pi shrinkage the estimator offers."""
    from oracle.formats import QJL_SHRINK, qjl_residual_estimate
    d, n = 128, 3000
    rng = np.random.default_rng(17)
    r = rng.standard_normal(d)
    r /= np.linalg.norm(r)
    e2, err = [], {1.0: [], QJL_SHRINK: []}
    for _ in range(n):
        S = rng.standard_normal((d, d))
        bits = (S @ r >= 0).astype(np.uint8)
        rh = qjl_residual_estimate(S, bits, 1.0)
        e2.append(rh @ rh)
        for s in err:
            dv = s * rh - r
            err[s].append(dv @ dv)
    kappa = np.pi / 2 + (d - 1) / d
    e2 = np.asarray(e2)
    assert abs(e2.mean() - kappa) < 4 * e2.std() / np.sqrt(n)
    for s, v in err.items():
        v = np.asarray(v)
        assert abs(v.mean() - (s * s * kappa - 2 * s + 1)) < 4 * v.std() / np.sqrt(n)
    assert np.mean(err[QJL_SHRINK]) < np.mean(err[1.0])


def norm_tree_row():
    """The row of tests/golden/norm_tree_row.txt."""
    x = np.zeros((1, D), np.float32)
    x[0, 0] = 8192.0
    for lane in (2, 4, 8, 16):
        x[0, 4 * lane] = 2.0
    for lane in range(1, 32, 2):
        x[0, 4 * lane:4 * lane + 3] = 1.0
    return x


def test_canonical_norm_tree_order_by_hand():
    """The fp32 norm follows the canonical addition order exactly: a row whose sum depends
    on the order gives the bits derived by hand from that order (golden file)."""
    from conftest import golden_lines
    fields = dict(ln.split()[:2] for ln in golden_lines("norm_tree_row.txt"))
    n = oracle.canonical_norm_fp32(norm_tree_row())
    assert int(n.view(np.uint32)[0]) == int(fields["n_bits"], 16)


def test_wht_signs_take_the_top_bit():
    """Sign j is -1 exactly when the top bit of splitmix64 output j is set: the golden
    outputs of seed 0 start 0xe220..., 0x6e78..., 0x06c4..., so the signs are -1, +1, +1."""
    from conftest import golden_lines
    outs = [int(v, 16) for v in golden_lines("splitmix64_seed0.txt")]
    assert [o >> 63 for o in outs] == [1, 0, 0]
    assert list(oracle.wht_signs(0, 3)) == [-1.0, 1.0, 1.0]


def test_prod3_layout_by_hand():
    """fp32 norm at bytes 0-3, fp32 residual norm at 4-7, 2-bit index of element j at bits
    2*(j%4) of byte 8 + j/4, QJL sign i at bit i%8 of byte 40 + i/8 (1 = +1)."""
    j = np.arange(D)
    idx = np.stack([j % 4, (j // 4) % 4]).astype(np.uint8)
    signs = np.stack([(j % 8 == 0), (j < 8) | (j % 8 == 7)]).astype(np.uint8)
    blk = oracle.pack_prod(np.array([2.0, 2.0], np.float32), np.array([0.5, 0.5], np.float32), idx, signs)
    for r in range(2):
        assert list(blk[r, 0:4]) == [0, 0, 0, 0x40]  # 2.0f = 0x40000000
        assert list(blk[r, 4:8]) == [0, 0, 0, 0x3F]  # 0.5f = 0x3F000000
    assert list(blk[0, 8:40]) == [0xE4] * 32  # elements 0..3 = 0, 1, 2, 3 -> 0b11100100
    assert list(blk[1, 8:40]) == [0x00, 0x55, 0xAA, 0xFF] * 8  # four equal codes per byte
    assert list(blk[0, 40:56]) == [0x01] * 16  # bit 0 of every byte
    assert list(blk[1, 40:56]) == [0xFF] + [0x80] * 15  # signs 0..7, then bit 7 of each byte
    n, g, back, sb = oracle.unpack_prod(blk)
    assert np.all(n == 2.0) and np.all(g == 0.5)
    assert np.array_equal(back, idx) and np.array_equal(sb, signs)
