"""CPU-only checks of the C-ABI library: it loads, exports every declared symbol, and its
host-side constructions (codebooks, rotations, QJL matrix, sizes, argument validation)
agree with the oracle.  No kernel is launched here."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tq():
    import __graft_entry__
    __graft_entry__.build()
    import compressed_attention_gb300 as m
    return m


def declared_functions():
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("tq_make_codebook", "tq_quantize_set_rows", "tq_decode_attention", "tq_dequantize"):
        assert required in names


def declared_arity():
    """Parameter count of every function the header declares."""
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = {}
    for m in re.finditer(r"\b(tq_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_matches_the_header(tq):
    """The Python binding declares every header function, with as many arguments."""
    decl, sig = declared_arity(), tq._SIGNATURES
    assert sorted(decl) == sorted(sig)
    assert {n: len(sig[n][1]) for n in decl} == decl


def test_library_exports_every_declared_symbol(tq):
    lib = ctypes.CDLL(tq.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []


@pytest.mark.parametrize("bits,kind", [(1, "quantile"), (2, "lloyd"), (3, "lloyd"), (4, "quantile"), (4, "lloyd"),
                                       (1, "sphere"), (2, "sphere"), (3, "sphere"), (4, "sphere")])
def test_host_codebook_matches_oracle(tq, bits, kind):
    c, b = tq.tq_make_codebook(bits, 128, kind)
    c32, b32 = oracle.stored_codebook(oracle.make_codebook(bits, 128, kind))
    assert np.max(np.abs(c - c32)) <= 1e-7
    assert np.max(np.abs(b - b32)) <= 1e-7 if bits > 1 else True


@pytest.mark.parametrize("seed", [0, 2, 3, 12345])
def test_host_dense_rotation_matches_oracle(tq, seed):
    pi = tq.tq_make_rotation("dense", seed).astype(np.float64)
    ref = oracle.dense_rotation(seed, 128)
    assert np.max(np.abs(pi - ref)) <= 1e-6
    assert np.max(np.abs(pi.T @ pi - np.eye(128))) <= 1e-6


@pytest.mark.parametrize("seed", [0, 5, 2**64 - 1])
def test_host_wht_signs_match_oracle(tq, seed):
    assert np.array_equal(tq.tq_make_rotation("wht", seed), oracle.wht_signs(seed, 128).astype(np.float32))


def test_host_qjl_matrix_matches_oracle(tq):
    S = tq.tq_make_qjl_matrix(1003)
    assert np.max(np.abs(S - oracle.qjl_matrix(1003, 128))) <= 1e-6


def test_sizes(tq):
    assert [tq.tq_row_bytes(f) for f in ("turbo4", "turbo3", "prod3", "vgroup2")] == [68, 56, 56, 48]
    assert tq.tq_cache_bytes("turbo4", 3) == 208  # 204 rounded up to 16
    assert tq.tq_cache_bytes("vgroup2", 1) == 48
    assert tq.lib.tq_row_bytes(9) == -1


def test_host_validation_errors(tq):
    lib = tq.lib
    c = np.zeros(16, np.float32)
    assert lib.tq_make_codebook(4, 64, 1, c.ctypes.data, None) == tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_make_codebook(5, 128, 1, c.ctypes.data, None) == tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_make_codebook(4, 128, 7, c.ctypes.data, None) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_make_codebook(4, 128, 1, None, None) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_quantize_set_rows(None, None, 0, 1, 128, None, None, 1, None) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_decode_attention(None, None, None, 0, None, None, None, 1, 1, 1, 1, 0.0, None, None,
                                   None, 0, None) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_decode_step(None, None, None, None, 0, 1, 128, None, None, 0, None, None, None, 1, 1, 1, 1,
                              0.0, None, None, 0, None) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_decode_step_host(None, None, None, 0, 1, None, 0, None, None, None, 1, 1, 1, 1,
                                   0.0, None, None, 0, None, 0, None) == tq.TQ_ERR_INVALID_ARG
    sz = ctypes.c_size_t(7)
    assert lib.tq_decode_step_host_staging_size(None, 0, 1, 0, 1, 1, ctypes.byref(sz)) == tq.TQ_ERR_INVALID_ARG
    assert sz.value == 7
    n = ctypes.c_int32(-1)
    assert lib.tq_decode_step_num_launches(None, None, 0, 1, 1, 1, 1, 1, ctypes.byref(n)) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_decode_step_num_launches(None, None, 0, 1, 1, 1, 1, 1, None) == tq.TQ_ERR_INVALID_ARG
    assert n.value == -1  # untouched on failure
    p = tq.tq_params(64, 0, 0, 0, 0, 0, 0, 0)
    h = ctypes.c_void_p()
    assert lib.tq_ctx_create(ctypes.byref(p), ctypes.byref(h)) == tq.TQ_ERR_UNSUPPORTED
    p = tq.tq_params(128, tq.TQ_FMT_PROD3, 0, tq.TQ_ROT_DENSE, 7, 7, 0, 0)
    assert lib.tq_ctx_create(ctypes.byref(p), ctypes.byref(h)) == tq.TQ_ERR_INVALID_ARG
    assert b"QJL seed" in lib.tq_last_error()
    p = tq.tq_params(128, tq.TQ_FMT_PROD3, 0, tq.TQ_ROT_DENSE, 7, 8, 2, 0)  # qjl_shrink not 0/1
    assert lib.tq_ctx_create(ctypes.byref(p), ctypes.byref(h)) == tq.TQ_ERR_INVALID_ARG
    p = tq.tq_params(128, tq.TQ_FMT_TURBO4, tq.TQ_CB_SPHERE + 1, tq.TQ_ROT_WHT, 7, 8, 0, 0)
    assert lib.tq_ctx_create(ctypes.byref(p), ctypes.byref(h)) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_status_string(tq.TQ_ERR_WORKSPACE) == b"workspace too small"


def test_decode_step_binding_rejects_mismatched_rows(tq):
    """The binding hands one source dtype and row stride to the C call, so new K and V
    rows that differ in either are refused before anything reaches the library."""
    import torch

    class Ctx:
        handle = None
    k = torch.zeros((4, 128), dtype=torch.bfloat16)
    for v in (torch.zeros((4, 128), dtype=torch.float32), torch.zeros((8, 128), dtype=torch.bfloat16)[::2]):
        with pytest.raises(ValueError):
            tq.tq_decode_step(Ctx, Ctx, k, v, None, None, None, None, None, 1, 4, 1, 8)


def test_static_area_size_matches_the_header(tq):
    """The binding reads the static scratch capacity from the library; it must equal the
    header's TQ_STATIC_WORKSPACE_BYTES."""
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    m = re.search(r"#define\s+TQ_STATIC_WORKSPACE_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m is not None
    assert tq.TQ_STATIC_WORKSPACE_BYTES == int(m.group(1)) << int(m.group(2))
