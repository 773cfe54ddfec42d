"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each one.

Each case monkeypatches one oracle function with a broken variant and asserts that
the corresponding pin fails; nothing here touches a GPU."""

import math

import numpy as np
import pytest

import oracle
import oracle.attention as att
import oracle.codebook as cb
import oracle.formats as fm
import oracle.rotation as rot
from conftest import golden_lines

D = 128


def printed_table():
    return np.array([float(v) for v in golden_lines("turbo4_centroids_d128.txt")])


def test_codebook_wrong_cell_index_is_caught(monkeypatch):
    good = cb.quantile_codebook(4, D)
    assert np.max(np.abs(good - printed_table())) <= 5e-5 + 1e-9

    def shifted(bits, d):  # off-by-one in the quantile cells
        K = 1 << bits
        sigma = 1 / math.sqrt(d)
        t = [cb.std_normal_quantile(min(k + 0.5, K) / K) for k in range(K + 1)]
        return np.array([sigma * cb._cond_mean_std(t[k], t[k + 1]) if t[k] < t[k + 1] else 0.0
                         for k in range(K)])

    bad = shifted(4, D)
    assert np.max(np.abs(bad - printed_table())) > 1e-3


def test_fwht_dropped_stage_is_caught():
    from scipy import linalg
    H = linalg.hadamard(D).astype(np.float64)

    def fwht_missing_last_stage(v):
        v = np.array(v, copy=True)
        h = 1
        while h < D // 2:
            w = v.reshape(v.shape[:-1] + (D // (2 * h), 2, h))
            a, b = w[..., 0, :].copy(), w[..., 1, :].copy()
            w[..., 0, :], w[..., 1, :] = a + b, a - b
            v = w.reshape(v.shape)
            h *= 2
        return v

    assert np.array_equal(rot.fwht(np.eye(D)), H.T)
    assert not np.array_equal(fwht_missing_last_stage(np.eye(D)), H.T)


def test_transposed_query_rotation_is_caught(monkeypatch):
    """Rotating q with Pi^T instead of Pi breaks compressed-domain == brute force."""
    kc = fm.Codec("turbo4", rotation="dense", rot_seed=3)
    x = np.random.default_rng(1).standard_normal((24, D)).astype(np.float32)
    kb = kc.encode(x)[0].reshape(1, 1, 24, -1)
    q = np.random.default_rng(2).standard_normal((1, 1, D))
    kh = kc.dequantize(kb.reshape(-1, 68)).reshape(1, 1, 24, D)
    ref, _ = oracle.attention_reference(q, kh, kh)
    monkeypatch.setattr(kc.rot, "forward", lambda u: np.asarray(u, dtype=np.float64) @ kc.rot.R)
    out, _ = att.attention_compressed_domain(q, kc, kb, kc, kb)
    assert np.max(np.abs(out - ref)) > 1e-3


def test_qjl_raw_signs_without_matrix_is_caught():
    """Section 2 bug 2 (signs used as raw +-1 instead of S^T sigma) breaks the brute-force
    prod score identity."""
    kc = fm.Codec("prod3", rotation="dense", rot_seed=3, qjl_seed=1003)
    x = np.random.default_rng(4).standard_normal((16, D)).astype(np.float32)
    blk, aux = kc.encode(x)
    good = kc.dequantize(blk)
    f = kc.fields(blk)
    raw = f["n"][:, None] * (kc.rot.inverse(f["y_hat"]) + (math.sqrt(math.pi / 2) / D) * f["gamma"][:, None] * f["sigma"])
    q = np.random.default_rng(5).standard_normal(D)
    assert np.max(np.abs(good @ q - raw @ q)) > 1e-2


def test_norm_without_square_is_caught():
    x = np.random.default_rng(6).standard_normal((10, D)).astype(np.float32)
    n = fm.canonical_norm_fp32(x)
    ref = np.linalg.norm(x.astype(np.float64), axis=1)
    assert np.max(np.abs(n - ref) / ref) < 4e-7
    bad = np.sqrt(np.abs(x).sum(1))
    assert np.max(np.abs(bad - ref) / ref) > 1e-2


def test_wrong_gqa_mapping_is_caught():
    wrong = [h % 8 for h in range(32)]
    right = [oracle.gqa_kv_head(h, 32, 8) for h in range(32)]
    assert wrong != right and right[:4] == [0, 0, 0, 0]


def test_prefill_mask_off_by_one_is_caught(monkeypatch):
    """A causal mask that stops one key early (or lets one key too many through) breaks
    the prefix-mean pin."""
    import test_oracle_prefill as pins

    def early(q, k_hat, v_hat, q_start, scale=None):
        q = np.asarray(q, dtype=np.float64)
        out = np.zeros(q.shape)
        for i in range(q.shape[1]):
            lens = [max(int(q_start[b]) + i, 1) for b in range(q.shape[0])]
            out[:, i], _ = att.attention_reference(q[:, i], k_hat, v_hat, lens, scale)
        return out

    def late(q, k_hat, v_hat, q_start, scale=None):
        q = np.asarray(q, dtype=np.float64)
        out = np.zeros(q.shape)
        for i in range(q.shape[1]):
            lens = [int(q_start[b]) + i + 2 for b in range(q.shape[0])]
            out[:, i], _ = att.attention_reference(q[:, i], k_hat, v_hat, lens, scale)
        return out

    for broken in (early, late):
        monkeypatch.setattr(oracle, "prefill_reference", broken)
        with pytest.raises(AssertionError):
            pins.test_identical_keys_give_prefix_means()


def test_vgroup_scale_zero_swapped_is_caught(monkeypatch):
    """A value dequantizer that reads the group's zero as its scale (and the scale as its
    zero) breaks the half-step reconstruction bound of the group quantizer."""
    from oracle.formats import Codec
    x = np.random.default_rng(9).standard_normal((300, D)).astype(np.float32) * 2.0
    codes, s16, z16 = oracle.encode_vgroup(x)
    blk = oracle.pack_vgroup(codes, s16, z16)
    s = np.repeat(s16.astype(np.float64), 32, axis=1)

    def within_bound(xh):
        return bool(np.all(np.abs(xh - x) <= 0.5 * s + 2e-3 * np.abs(x).max()))

    assert within_bound(Codec("vgroup2").dequantize(blk))
    good = fm.unpack_vgroup

    def swapped(blocks):
        c, sc, ze = good(blocks)
        return c, ze, sc

    monkeypatch.setattr(fm, "unpack_vgroup", swapped)
    assert not within_bound(Codec("vgroup2").dequantize(blk))


def test_turbo3_sign_bit_order_is_caught():
    """Sign bits stored most-significant first in their byte (instead of bit j % 8 for
    element j) contradict the layout the pages print, which the by-hand pin checks."""
    idx = (np.arange(D) % 8).astype(np.uint8)[None, :]
    good = oracle.pack_turbo3(np.array([1.0], np.float32), idx)
    bad = good.copy()
    for c in range(4):
        sl = slice(14 * c + 10, 14 * c + 14)
        bad[:, sl] = np.packbits(np.unpackbits(bad[:, sl], axis=1, bitorder="little"), axis=1, bitorder="big")
    for blk, ok in ((good, True), (bad, False)):
        assert (list(blk[0, 10:14]) == [0xF0] * 4) == ok
        assert np.array_equal(oracle.unpack_turbo3(blk)[1], idx) == ok


def test_prod3_sign_bits_reversed_is_caught(monkeypatch):
    """QJL sign i stored at bit 7 - i%8 (in both the packer and the unpacker, so a round
    trip still passes) contradicts the by-hand byte layout."""
    import test_oracle_formats as pins
    good_pack, good_unpack = fm.pack_prod, fm.unpack_prod

    def rev(b):
        return np.packbits(np.unpackbits(b, axis=1, bitorder="little"), axis=1, bitorder="big")

    def pack(n32, gamma32, idx, sign_bits):
        out = good_pack(n32, gamma32, idx, sign_bits)
        out[:, 40:56] = rev(out[:, 40:56])
        return out

    def unpack(blocks):
        b = np.array(blocks, dtype=np.uint8, copy=True)
        b[:, 40:56] = rev(b[:, 40:56])
        return good_unpack(b)

    for name, f in (("pack_prod", pack), ("unpack_prod", unpack)):
        monkeypatch.setattr(oracle, name, f)
        monkeypatch.setattr(fm, name, f)
    with pytest.raises(AssertionError):
        pins.test_prod3_layout_by_hand()


def test_prod3_norm_and_residual_norm_swapped_is_caught(monkeypatch):
    import test_oracle_formats as pins
    good_pack = fm.pack_prod
    monkeypatch.setattr(oracle, "pack_prod", lambda n, g, i, s: good_pack(g, n, i, s))
    with pytest.raises(AssertionError):
        pins.test_prod3_layout_by_hand()


def test_wht_sign_from_low_bit_is_caught(monkeypatch):
    """Taking bit 0 of each splitmix64 output instead of the top bit passes the +-1 and
    balance checks but not the signs the golden outputs fix."""
    import test_oracle_formats as pins

    def low_bit(seed, d):
        return np.where((rot.splitmix64(seed, d) & np.uint64(1)) == 1, -1.0, 1.0)

    monkeypatch.setattr(oracle, "wht_signs", low_bit)
    with pytest.raises(AssertionError):
        pins.test_wht_signs_take_the_top_bit()


@pytest.mark.parametrize("order", ["elements_left_to_right", "adjacent_lanes_first", "fp64_then_round"])
def test_norm_in_another_order_is_caught(monkeypatch, order):
    """Any summation order other than the canonical tree changes the norm of the golden
    row; each plausible alternative is planted and caught."""
    import test_oracle_formats as pins

    def other(x):
        x32 = np.asarray(x, dtype=np.float32)
        sq = x32 * x32
        if order == "elements_left_to_right":
            s = np.zeros(len(x32), np.float32)
            for j in range(x32.shape[1]):
                s = (s + sq[:, j]).astype(np.float32)
        elif order == "adjacent_lanes_first":
            p = (sq[:, 0::4] + sq[:, 1::4]) + (sq[:, 2::4] + sq[:, 3::4])
            while p.shape[1] > 1:
                p = (p[:, 0::2] + p[:, 1::2]).astype(np.float32)
            s = p[:, 0]
        else:
            s = (x32.astype(np.float64) ** 2).sum(axis=1).astype(np.float32)
        return np.sqrt(s).astype(np.float32)

    monkeypatch.setattr(oracle, "canonical_norm_fp32", other)
    with pytest.raises(AssertionError):
        pins.test_canonical_norm_tree_order_by_hand()
