"""Helpers shared by the GPU parity tests (imported lazily by ``-m gpu`` tests only)."""

import numpy as np

import synth

ATOL = 2e-3   # max abs error of scores and outputs against the oracle
RTOL = 1e-3   # per (b, h): ||o_gpu - o_ref|| / ||o_ref||
BAND = 1e-5   # dense rotation: indices may differ only this close to a boundary


def lib():
    import __graft_entry__
    __graft_entry__.build()
    import compressed_attention_gb300 as tq
    return tq


def torch_rows(x32, dtype):
    """fp32 numpy rows -> CUDA tensor of dtype ('f32' or 'bf16'), plus the exact fp32 values."""
    import torch
    if dtype == "bf16":
        bits = synth.bf16_bits(x32)
        t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()
        return t, synth.bf16_to_f32(bits)
    if dtype == "f16":
        h = x32.astype(np.float16)
        return torch.from_numpy(h.copy()).cuda(), h.astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).cuda(), np.asarray(x32, np.float32)


def to_host_bytes(cache, n_rows, row_bytes):
    return cache.cpu().numpy()[: n_rows * row_bytes].reshape(n_rows, row_bytes)


def check_outputs(out_gpu, out_ref, atol=ATOL, rtol=RTOL):
    out_gpu = np.asarray(out_gpu, np.float64)
    out_ref = np.asarray(out_ref, np.float64)
    err = np.abs(out_gpu - out_ref)
    assert np.all(np.isfinite(out_gpu)), "non-finite output"
    assert err.max() <= atol, f"max abs error {err.max():.3e} > {atol}"
    num = np.linalg.norm((out_gpu - out_ref).reshape(-1, out_ref.shape[-1]), axis=1)
    den = np.linalg.norm(out_ref.reshape(-1, out_ref.shape[-1]), axis=1)
    rel = num / np.maximum(den, 1e-30)
    assert rel.max() <= rtol, f"max relative error {rel.max():.3e} > {rtol}"
    return err.max(), rel.max()


def band_ok(idx_gpu, idx_ref, y_ref, b32, band=BAND):
    """Indices may differ only by one cell and only where the oracle coordinate lies within
    `band` of the boundary between the two cells."""
    diff = idx_gpu.astype(np.int64) != idx_ref.astype(np.int64)
    if not diff.any():
        return True, 0
    lo = np.minimum(idx_gpu, idx_ref)[diff].astype(np.int64)
    step = np.abs(idx_gpu.astype(np.int64) - idx_ref.astype(np.int64))[diff]
    if np.any(step != 1):
        return False, int(diff.sum())
    dist = np.abs(y_ref[diff] - b32.astype(np.float64)[lo])
    return bool(np.all(dist < band)), int(diff.sum())


def norm_byte_mask(fmt):
    """Byte positions holding a norm field in one packed row."""
    m = np.zeros({"turbo4": 68, "turbo3": 56, "prod3": 56, "vgroup2": 48}[fmt], bool)
    if fmt == "turbo4":
        m[:4] = True
    elif fmt == "turbo3":
        for c in range(4):
            m[14 * c:14 * c + 2] = True
    elif fmt == "prod3":
        m[:8] = True
    return m


def rows_equal_nan_aware(got, ref, fmt):
    """Bit equality of packed rows, except that a NaN norm may carry any NaN payload
    (IEEE leaves the payload of a generated NaN to the implementation)."""
    bad = np.nonzero(np.any(got != ref, axis=1))[0]
    if bad.size == 0 or fmt == "vgroup2":
        return bad
    mask = norm_byte_mask(fmt)
    keep = []
    for r in bad:
        if np.any(got[r, ~mask] != ref[r, ~mask]):
            keep.append(r)
            continue
        if fmt == "turbo3":
            g = got[r, mask].copy().view("<f2")
            e = ref[r, mask].copy().view("<f2")
        else:
            g = got[r, mask].copy().view("<f4")
            e = ref[r, mask].copy().view("<f4")
        if not np.all((g == e) | (np.isnan(g) & np.isnan(e))):
            keep.append(r)
    return np.array(keep, dtype=np.int64)
