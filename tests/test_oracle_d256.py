"""Pins of the oracle at head dimension 256 (turbo4 only).

A d = 256 turbo4 row is two consecutive 68-byte blocks (the 128-element block of the
turbo4 format), block c holding elements 128c .. 128c+127 of the rotated row and the
row's norm; readers scale each block by its own stored norm."""

import math

import numpy as np
import pytest

import oracle
from conftest import golden_lines
from oracle.formats import Codec

D = 256


def test_canonical_norm_tree_d256_by_hand():
    fields = dict(ln.split()[:2] for ln in golden_lines("norm_tree_row_d256.txt"))
    x = np.zeros((1, D), np.float32)
    x[0, 0] = 8192.0
    for lane in (2, 4, 8, 16):
        x[0, 8 * lane] = 2.0
    for lane in range(1, 32, 2):
        x[0, 8 * lane:8 * lane + 3] = 1.0
    n = oracle.canonical_norm_fp32(x)
    assert int(n.view(np.uint32)[0]) == int(fields["n_bits"], 16)
    # and the tree is a sum of squares: random rows agree with fp64 to fp32 accuracy
    r = np.random.default_rng(0).standard_normal((200, D)).astype(np.float32) * 3
    ref = np.linalg.norm(r.astype(np.float64), axis=1)
    assert np.max(np.abs(oracle.canonical_norm_fp32(r) - ref) / ref) < 5e-7


def test_codebook_scales_with_one_over_sqrt_d():
    """Centroids of N(0, 1/d): c_k(d) = c_k(1) / sqrt(d), so the d = 256 table is the
    d = 128 one divided by sqrt(2) (and the printed d = 128 table pins that one)."""
    c128 = oracle.make_codebook(4, 128, "quantile")
    c256 = oracle.make_codebook(4, D, "quantile")
    assert np.max(np.abs(c256 * math.sqrt(2.0) - c128)) < 1e-12


def test_wht_256_is_the_sylvester_matrix_and_rotations_are_orthogonal():
    from scipy import linalg
    H = linalg.hadamard(D).astype(np.float64)
    assert np.array_equal(oracle.fwht(np.eye(D)), H.T)
    R = oracle.wht_rotation_matrix(oracle.wht_signs(5, D))
    assert np.max(np.abs(R @ R.T - np.eye(D))) < 1e-12
    Pi = oracle.dense_rotation(7, D).astype(np.float32).astype(np.float64)
    assert np.max(np.abs(Pi.T @ Pi - np.eye(D))) < 1e-6


def test_d256_row_layout_by_hand():
    """Block 0 = norm + nibbles of elements 0..127, block 1 = norm + elements 128..255."""
    idx = np.zeros((1, D), np.uint8)
    idx[0, :128] = np.arange(128) % 16
    idx[0, 128:] = 15 - np.arange(128) % 16
    rows = oracle.pack_turbo4_rows(np.array([2.0], np.float32), idx)
    assert rows.shape == (1, 136)
    assert list(rows[0, 0:4]) == [0, 0, 0, 0x40] and list(rows[0, 68:72]) == [0, 0, 0, 0x40]
    assert rows[0, 4] == 0x10 and rows[0, 5] == 0x32      # elements 0, 1 | 2, 3
    assert rows[0, 72] == 0xEF and rows[0, 73] == 0xCD    # elements 128 (15), 129 (14) | 130, 131
    norms, back = oracle.unpack_turbo4_rows(rows, D)
    assert np.all(norms == 2.0) and np.array_equal(back, idx)


@pytest.mark.parametrize("rotation", ["wht", "dense"])
def test_d256_encode_is_nearest_centroid_and_reconstructs(rotation):
    codec = Codec("turbo4", d=D, rotation=rotation, rot_seed=11)
    x = (np.random.default_rng(4).standard_normal((400, D)) * 2.0).astype(np.float32)
    blk, aux = codec.encode(x)
    assert blk.shape == (400, 136)
    u = x.astype(np.float64) / np.linalg.norm(x.astype(np.float64), axis=1, keepdims=True)
    assert np.max(np.abs(codec.rot.forward(u) - aux["y"])) < 2e-6
    c = codec.c32.astype(np.float64)
    assert np.array_equal(np.argmin(np.abs(aux["y"][..., None] - c), axis=-1), aux["idx"])
    # per-coordinate distortion d * MSE of the 16-level quantile table (the same at any d)
    xh = codec.dequantize(blk)
    rel = np.sum((xh - x) ** 2, axis=1) / np.sum(x.astype(np.float64) ** 2, axis=1)
    assert abs(rel.mean() - 0.0203) / 0.0203 < 0.06


def test_d256_brute_force_equals_compressed_domain_with_own_block_norms():
    """Dequantize-then-softmax equals the compressed-domain path at d = 256, also when the
    two blocks of a row carry different norms (each block scales by its own)."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, L = 2, 4, 2, 40
    kc = Codec("turbo4", d=D, rotation="dense", rot_seed=21)
    vc = Codec("turbo4", d=D, rotation="wht", rot_seed=22)
    kb = kc.encode(rng.standard_normal((B * Hkv * L, D)).astype(np.float32))[0]
    vb = vc.encode(rng.standard_normal((B * Hkv * L, D)).astype(np.float32))[0].copy()
    n1 = vb[:, 68:72].copy().view("<f4") * rng.uniform(0.5, 2.0, (len(vb), 1)).astype(np.float32)
    vb[:, 68:72] = n1.view(np.uint8)
    q = rng.standard_normal((B, Hq, D))
    kh = kc.dequantize(kb).reshape(B, Hkv, L, D)
    vh = vc.dequantize(vb).reshape(B, Hkv, L, D)
    ref, s_ref = oracle.attention_reference(q, kh, vh, [L, 17])
    out, s = oracle.attention_compressed_domain(q, kc, kb.reshape(B, Hkv, L, -1), vc, vb.reshape(B, Hkv, L, -1),
                                                [L, 17], n_chunks=3)
    assert np.max(np.abs(out - ref)) < 1e-10
    m = ~np.isnan(s_ref)
    assert np.max(np.abs(s[m] - s_ref[m])) < 1e-10
    # the second block's own norm matters: a reader using block 0's norm for both differs
    wrong = vb.copy()
    wrong[:, 68:72] = wrong[:, 0:4]
    assert np.max(np.abs(vc.dequantize(wrong) - vc.dequantize(vb))) > 1e-2
