"""Thin Python binding of the GB300 compressed-KV library (``include/tq.h``).

Every function here only marshals arguments for the C ABI of ``lib/libtq.so``:
device buffers are passed as torch tensors (or raw integer addresses), streams
default to torch's current CUDA stream.  All computation runs in the library's
CUDA kernels; if the library has not been built, importing this package raises
ImportError instead of falling back to anything else.

Build the library with ``python compressed_attention_gb300/_build.py`` (or
``__graft_entry__.build()``); the build script does not import this package.
"""

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libtq.so")

D = 128

# tq_status
TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_ALIGNMENT, TQ_ERR_CUDA, TQ_ERR_ALLOC, TQ_ERR_WORKSPACE = range(7)
# tq_format
TQ_FMT_TURBO4, TQ_FMT_TURBO3, TQ_FMT_PROD3, TQ_FMT_VGROUP2 = range(4)
# tq_codebook_kind
TQ_CB_DEFAULT, TQ_CB_QUANTILE, TQ_CB_LLOYD, TQ_CB_SPHERE = range(4)
# tq_rotation_kind
TQ_ROT_WHT, TQ_ROT_DENSE = range(2)
# tq_dtype
TQ_DTYPE_F32, TQ_DTYPE_BF16, TQ_DTYPE_F16 = range(3)

FORMATS = {"turbo4": TQ_FMT_TURBO4, "turbo3": TQ_FMT_TURBO3, "prod3": TQ_FMT_PROD3, "vgroup2": TQ_FMT_VGROUP2}
ROTATIONS = {"wht": TQ_ROT_WHT, "dense": TQ_ROT_DENSE}
CODEBOOKS = {None: TQ_CB_DEFAULT, "default": TQ_CB_DEFAULT, "quantile": TQ_CB_QUANTILE, "lloyd": TQ_CB_LLOYD,
             "sphere": TQ_CB_SPHERE}


class TQError(RuntimeError):
    def __init__(self, status, func, detail):
        self.status = status
        super().__init__(f"{func} failed with status {status}: {detail}")


class tq_params(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("format", ctypes.c_int32), ("codebook", ctypes.c_int32),
                ("rotation", ctypes.c_int32), ("rot_seed", ctypes.c_uint64), ("qjl_seed", ctypes.c_uint64),
                ("qjl_shrink", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_vp, _i32, _i64, _u64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                                    ctypes.c_float, ctypes.c_size_t)

_SIGNATURES = {
    "tq_make_codebook": (_i32, [_i32, _i32, _i32, _vp, _vp]),
    "tq_make_rotation": (_i32, [_i32, _i32, _u64, _vp]),
    "tq_make_qjl_matrix": (_i32, [_i32, _u64, _vp]),
    "tq_row_bytes": (_i64, [_i32]),
    "tq_cache_bytes": (_sz, [_i32, _i64]),
    "tq_status_string": (ctypes.c_char_p, [_i32]),
    "tq_last_error": (ctypes.c_char_p, []),
    "tq_ctx_create": (_i32, [ctypes.POINTER(tq_params), ctypes.POINTER(_vp)]),
    "tq_ctx_destroy": (_i32, [_vp]),
    "tq_ctx_device_status": (_i32, [_vp, ctypes.POINTER(ctypes.c_int32), _i32]),
    "tq_quantize_set_rows": (_i32, [_vp, _vp, _i32, _i64, _i64, _vp, _vp, _i64, _vp]),
    "tq_dequantize": (_i32, [_vp, _vp, _i64, _i32, _vp, _vp]),
    "tq_decode_workspace_size": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, ctypes.POINTER(_sz)]),
    "tq_decode_num_splits": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, ctypes.POINTER(_i32)]),
    "tq_decode_num_launches": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, ctypes.POINTER(_i32)]),
    "tq_decode_step_num_launches": (_i32, [_vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32, ctypes.POINTER(_i32)]),
    "tq_decode_step": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i64, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32,
                              _i32, _i32, _f32, _vp, _vp, _sz, _vp]),
    "tq_decode_step_host": (_i32, [_vp, _vp, _vp, _i32, _i64, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                   _f32, _vp, _vp, _sz, _vp, _sz, _vp]),
    "tq_decode_step_host_staging_size": (_i32, [_vp, _i32, _i64, _i32, _i32, _i32, ctypes.POINTER(_sz)]),
    "tq_decode_attention": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _f32,
                                   _vp, _vp, _vp, _sz, _vp]),
    "tq_decode_prepare_q": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _sz, _vp]),
    "tq_decode_partial": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
    "tq_decode_combine": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
    "tq_decode_partial_merge": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
    "tq_decode_attention_static": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _f32,
                                          _vp, _vp]),
    "tq_static_workspace_bytes": (_sz, []),
    "tq_test_decode_wait_timeout": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _sz, _vp]),
    "tq_test_ctx_set_device": (_i32, [_vp, _i32]),
    "tq_store_create": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, ctypes.POINTER(_vp)]),
    "tq_store_destroy": (_i32, [_vp]),
    "tq_store_append": (_i32, [_vp, _vp, _vp, _i32, _vp]),
    "tq_store_state": (_i32, [_vp, ctypes.POINTER(_i64), ctypes.POINTER(_i64), ctypes.POINTER(_vp),
                              ctypes.POINTER(_vp)]),
    "tq_store_workspace_size": (_i32, [_vp, _i32, ctypes.POINTER(_sz)]),
    "tq_store_decode": (_i32, [_vp, _vp, _i32, _i32, _f32, _vp, _vp, _sz, _vp]),
    "tq_prefill_workspace_size": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_sz)]),
    "tq_prefill_attention": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                    _f32, _vp, _vp, _sz, _vp]),
    "tq_prefill_prepare_q": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _sz, _vp]),
    "tq_prefill_partial": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _sz, _vp]),
    "tq_prefill_combine": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python compressed_attention_gb300/_build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def _check(status, func):
    if status != TQ_OK:
        raise TQError(status, func, lib.tq_last_error().decode())


def _ptr(x):
    if x is None:
        return None
    dp = getattr(x, "data_ptr", None)  # a tensor (the common case first)
    if dp is not None:
        return dp()
    if isinstance(x, int):
        return x
    if hasattr(x, "ctypes"):  # numpy array (host)
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x).__name__}")


_TORCH = None  # (torch module, CUDA available, dtype -> library code), looked up once


def _torch():
    global _TORCH
    if _TORCH is None:
        import torch
        _TORCH = (torch, torch.cuda.is_available(),
                  {torch.float32: TQ_DTYPE_F32, torch.bfloat16: TQ_DTYPE_BF16, torch.float16: TQ_DTYPE_F16})
    return _TORCH


def _stream(stream):
    if stream is None:
        torch, cuda, _ = _torch()
        if not cuda:
            return None
        # the raw handle of the current stream, without building a Stream object
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device()) or None
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _torch_dtype_code(dt):
    return _torch()[2][dt]


def _dtype_code(t):
    return _torch_dtype_code(t.dtype)


# --------------------------------------------------------------------------- host only

def tq_make_codebook(bits, d=D, kind="quantile"):
    """(centroids float32[2^bits], boundaries float32[2^bits - 1]) built on the host."""
    import numpy as np
    K = 1 << bits
    c = np.zeros(K, np.float32)
    b = np.zeros(max(K - 1, 1), np.float32)
    _check(lib.tq_make_codebook(bits, d, CODEBOOKS[kind], c.ctypes.data, b.ctypes.data), "tq_make_codebook")
    return c, b[:K - 1]


def tq_make_rotation(kind, seed, d=D):
    """Dense: float32 [d, d] Pi (y = Pi u).  WHT: float32 [d] signs."""
    import numpy as np
    out = np.zeros((d, d) if kind == "dense" else (d,), np.float32)
    _check(lib.tq_make_rotation(ROTATIONS[kind], d, seed, out.ctypes.data), "tq_make_rotation")
    return out


def tq_make_qjl_matrix(seed, d=D):
    import numpy as np
    out = np.zeros((d, d), np.float32)
    _check(lib.tq_make_qjl_matrix(d, seed, out.ctypes.data), "tq_make_qjl_matrix")
    return out


def tq_row_bytes(fmt):
    return int(lib.tq_row_bytes(FORMATS.get(fmt, fmt)))


def tq_cache_bytes(fmt, n_rows):
    return int(lib.tq_cache_bytes(FORMATS.get(fmt, fmt), n_rows))


# --------------------------------------------------------------------------- contexts

class Ctx:
    """Owns one tq_ctx (codebook, rotation, QJL matrix on the current device)."""

    def __init__(self, fmt, rotation="wht", rot_seed=0, qjl_seed=0, codebook=None, d=D, qjl_shrink=False):
        self.fmt = fmt
        self.rotation = rotation
        self.rot_seed = rot_seed
        self.qjl_seed = qjl_seed
        p = tq_params(d, FORMATS[fmt], CODEBOOKS[codebook], ROTATIONS[rotation], rot_seed, qjl_seed,
                      int(bool(qjl_shrink)), 0)
        h = _vp()
        _check(lib.tq_ctx_create(ctypes.byref(p), ctypes.byref(h)), "tq_ctx_create")
        self.handle = h.value
        self.d = d
        # a row of head dimension 256 is two 128-element turbo4 blocks
        self.row_bytes = tq_row_bytes(fmt) * d // D

    def close(self):
        if getattr(self, "handle", None):
            lib.tq_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tq_ctx_create(fmt, rotation="wht", rot_seed=0, qjl_seed=0, codebook=None, d=D):
    return Ctx(fmt, rotation, rot_seed, qjl_seed, codebook, d)


def tq_ctx_destroy(ctx):
    ctx.close()


def tq_ctx_device_status(ctx, clear=True):
    v = ctypes.c_int32(0)
    _check(lib.tq_ctx_device_status(ctx.handle, ctypes.byref(v), int(clear)), "tq_ctx_device_status")
    return v.value


# --------------------------------------------------------------------------- write / read

def tq_quantize_set_rows(ctx, src, dst_cache, row_ids=None, n_rows=None, stream=None):
    """Quantize rows of ``src`` ([n, d] fp32/bf16 CUDA tensor) into ``dst_cache`` (uint8 CUDA
    tensor of packed rows) at slots ``row_ids`` (int64 CUDA tensor) or 0..n-1."""
    n = src.shape[0] if n_rows is None else n_rows
    stride = src.stride(0) if src.dim() == 2 else D
    dst_rows = dst_cache.numel() // ctx.row_bytes
    _check(lib.tq_quantize_set_rows(ctx.handle, _ptr(src), _dtype_code(src), n, stride, _ptr(row_ids),
                                    _ptr(dst_cache), dst_rows, _stream(stream)), "tq_quantize_set_rows")


def tq_dequantize(ctx, cache, n_rows, dst, unrotate=True, stream=None):
    _check(lib.tq_dequantize(ctx.handle, _ptr(cache), n_rows, int(unrotate), _ptr(dst), _stream(stream)),
           "tq_dequantize")


def tq_decode_workspace_size(k_ctx, v_ctx, B, Hq, Hkv, L):
    n = _sz(0)
    _check(lib.tq_decode_workspace_size(k_ctx.handle, v_ctx.handle, B, Hq, Hkv, L, ctypes.byref(n)),
           "tq_decode_workspace_size")
    return n.value


def tq_decode_step(k_ctx, v_ctx, new_k, new_v, q, k_cache, v_cache, out, workspace, B, Hq, Hkv, L,
                   row_ids=None, seq_lens=None, scale=0.0, stream=None):
    """SET_ROWS of the step's new K / V rows ([n, 128] tensors, rows at slots row_ids of the
    [B][Hkv][L] caches), then decode attention over the updated caches."""
    if new_v.dtype != new_k.dtype or new_v.shape != new_k.shape or new_v.stride() != new_k.stride():
        raise ValueError("new_k and new_v must have one dtype, shape and row stride")
    n = new_k.shape[0] if new_k.dim() == 2 else new_k.numel() // D
    qp, qd = _q_args(q)
    _check(lib.tq_decode_step(k_ctx.handle, v_ctx.handle, _ptr(new_k), _ptr(new_v), _dtype_code(new_k), n,
                              new_k.stride(-2) if new_k.dim() >= 2 else D, _ptr(row_ids), qp, qd, _ptr(k_cache),
                              _ptr(v_cache), _ptr(seq_lens), B, Hq, Hkv, L, scale, _ptr(out), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)), "tq_decode_step")


def tq_decode_step_host_staging_size(k_ctx, src_dtype, n_rows, q_dtype, B, Hq):
    """Device staging bytes tq_decode_step_host needs (torch dtypes of the rows and of q)."""
    n = _sz(0)
    _check(lib.tq_decode_step_host_staging_size(k_ctx.handle, _torch_dtype_code(src_dtype), n_rows,
                                                _torch_dtype_code(q_dtype), B, Hq, ctypes.byref(n)),
           "tq_decode_step_host_staging_size")
    return n.value


def pack_step_inputs(new_k, new_v, q):
    """One pinned host buffer holding new_k, new_v and q back to back (tq_decode_step_host's
    input layout), and the host views of the three parts in it."""
    import torch
    parts = [new_k, new_v, q]
    sizes = [t.numel() * t.element_size() for t in parts]
    buf = torch.empty(sum(sizes), dtype=torch.uint8, pin_memory=True)
    views, off = [], 0
    for t, n in zip(parts, sizes):
        v = buf[off:off + n].view(t.dtype).view(t.shape)
        v.copy_(t.detach().cpu())
        views.append(v)
        off += n
    return buf, views


def tq_decode_step_host(k_ctx, v_ctx, inputs, src_dtype, n_rows, q_dtype, out, row_ids, k_cache, v_cache, staging,
                        workspace, B, Hq, Hkv, L, seq_lens=None, scale=0.0, stream=None):
    """tq_decode_step with host buffers: ``inputs`` a (pinned) host buffer holding the new K
    rows, the new V rows ([n_rows, d] of src_dtype each) and q ([B, Hq, d] of q_dtype) back
    to back (pack_step_inputs), ``out`` fp32 [B, Hq, d] in host memory; one C call copies
    the inputs in, runs the step on the device staging area and copies the output back, on
    the stream, without waiting."""
    _check(lib.tq_decode_step_host(k_ctx.handle, v_ctx.handle, _ptr(inputs), _torch_dtype_code(src_dtype), n_rows,
                                   _ptr(row_ids), _torch_dtype_code(q_dtype), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(seq_lens), B, Hq, Hkv, L, scale, _ptr(out), _ptr(staging),
                                   staging.numel() * staging.element_size(), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "tq_decode_step_host")


def tq_decode_step_num_launches(k_ctx, v_ctx, src_dtype, n_rows, B, Hq, Hkv, L):
    """Kernels one tq_decode_step call launches (``src_dtype`` a torch dtype)."""
    import torch
    n = _i32(0)
    code = TQ_DTYPE_BF16 if src_dtype == torch.bfloat16 else TQ_DTYPE_F32
    _check(lib.tq_decode_step_num_launches(k_ctx.handle, v_ctx.handle, code, n_rows, B, Hq, Hkv, L,
                                           ctypes.byref(n)), "tq_decode_step_num_launches")
    return n.value


def tq_decode_num_launches(k_ctx, v_ctx, B, Hq, Hkv, L):
    n = _i32(0)
    _check(lib.tq_decode_num_launches(k_ctx.handle, v_ctx.handle, B, Hq, Hkv, L, ctypes.byref(n)),
           "tq_decode_num_launches")
    return n.value


def tq_decode_num_splits(k_ctx, v_ctx, B, Hq, Hkv, L):
    n = _i32(0)
    _check(lib.tq_decode_num_splits(k_ctx.handle, v_ctx.handle, B, Hq, Hkv, L, ctypes.byref(n)),
           "tq_decode_num_splits")
    return n.value


def _q_args(q):
    return _ptr(q), _dtype_code(q)


def tq_decode_attention(k_ctx, v_ctx, q, k_cache, v_cache, out, workspace, B, Hq, Hkv, L,
                        seq_lens=None, scale=0.0, scores=None, stream=None):
    qp, qd = _q_args(q)
    _check(lib.tq_decode_attention(k_ctx.handle, v_ctx.handle, qp, qd, _ptr(k_cache), _ptr(v_cache),
                                   _ptr(seq_lens), B, Hq, Hkv, L, scale, _ptr(out), _ptr(scores),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)), "tq_decode_attention")


def tq_prefill_workspace_size(k_ctx, v_ctx, B, T, Hq, Hkv, L):
    n = _sz(0)
    _check(lib.tq_prefill_workspace_size(k_ctx.handle, v_ctx.handle, B, T, Hq, Hkv, L, ctypes.byref(n)),
           "tq_prefill_workspace_size")
    return n.value


def tq_prefill_attention(k_ctx, v_ctx, q, k_cache, v_cache, q_start, out, workspace, B, T, Hq, Hkv, L,
                         scale=0.0, stream=None):
    """Causal attention of T chunk queries per sequence (q [B, T, Hq, 128], query i of
    sequence b at position q_start[b] + i) over the packed caches."""
    qp, qd = _q_args(q)
    _check(lib.tq_prefill_attention(k_ctx.handle, v_ctx.handle, qp, qd, _ptr(k_cache), _ptr(v_cache),
                                    _ptr(q_start), B, T, Hq, Hkv, L, scale, _ptr(out), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "tq_prefill_attention")


def _wsb(workspace):
    return workspace.numel() * workspace.element_size()


def tq_prefill_prepare_q(k_ctx, v_ctx, q, workspace, B, T, Hq, Hkv, L, scale=0.0, stream=None):
    qp, qd = _q_args(q)
    _check(lib.tq_prefill_prepare_q(k_ctx.handle, v_ctx.handle, qp, qd, B, T, Hq, Hkv, L, scale,
                                    _ptr(workspace), _wsb(workspace), _stream(stream)), "tq_prefill_prepare_q")


def tq_prefill_partial(k_ctx, v_ctx, k_cache, v_cache, q_start, workspace, B, T, Hq, Hkv, L, stream=None):
    _check(lib.tq_prefill_partial(k_ctx.handle, v_ctx.handle, _ptr(k_cache), _ptr(v_cache), _ptr(q_start),
                                  B, T, Hq, Hkv, L, _ptr(workspace), _wsb(workspace), _stream(stream)),
           "tq_prefill_partial")


def tq_prefill_combine(k_ctx, v_ctx, out, workspace, B, T, Hq, Hkv, L, stream=None):
    _check(lib.tq_prefill_combine(k_ctx.handle, v_ctx.handle, B, T, Hq, Hkv, L, _ptr(out), _ptr(workspace),
                                  _wsb(workspace), _stream(stream)), "tq_prefill_combine")


class _DeviceBytes:
    """A device byte range seen through the CUDA array interface (no copy, no ownership)."""

    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False),
                                         "version": 3}


class Store:
    """A ring-buffer capture + block-append store (tq_store_*): recent tokens exact in a
    device ring, older ones compressed in the store's caches; decode attends over both."""

    def __init__(self, k_ctx, v_ctx, B, Hkv, L, ring_tokens):
        self.k_ctx, self.v_ctx, self.B, self.Hkv, self.L = k_ctx, v_ctx, B, Hkv, L
        h = _vp()
        _check(lib.tq_store_create(k_ctx.handle, v_ctx.handle, B, Hkv, L, ring_tokens, ctypes.byref(h)),
               "tq_store_create")
        self.handle = h.value

    def close(self):
        if self.handle:
            lib.tq_store_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def append(self, k_new, v_new, stream=None):
        """k_new, v_new: bf16 [B, Hkv, n, 128] device tensors."""
        n = k_new.shape[2]
        _check(lib.tq_store_append(self.handle, _ptr(k_new), _ptr(v_new), n, _stream(stream)), "tq_store_append")

    def state(self):
        n, f, kc, vc = _i64(0), _i64(0), _vp(), _vp()
        _check(lib.tq_store_state(self.handle, ctypes.byref(n), ctypes.byref(f), ctypes.byref(kc), ctypes.byref(vc)),
               "tq_store_state")
        return n.value, f.value, kc.value, vc.value

    def cache_bytes(self, which):
        """The compressed cache (which = "k" or "v") as a uint8 device tensor (a view)."""
        import torch
        _, _, kc, vc = self.state()
        ctx = self.k_ctx if which == "k" else self.v_ctx
        nbytes = tq_cache_bytes(ctx.fmt, self.B * self.Hkv * self.L)
        return torch.as_tensor(_DeviceBytes(kc if which == "k" else vc, nbytes), device="cuda")

    def workspace_size(self, Hq):
        n = _sz(0)
        _check(lib.tq_store_workspace_size(self.handle, Hq, ctypes.byref(n)), "tq_store_workspace_size")
        return n.value

    def decode(self, q, out, workspace, Hq, scale=0.0, stream=None):
        qp, qd = _q_args(q)
        _check(lib.tq_store_decode(self.handle, qp, qd, Hq, scale, _ptr(out), _ptr(workspace), _wsb(workspace),
                                   _stream(stream)), "tq_store_decode")


TQ_STATIC_WORKSPACE_BYTES = lib.tq_static_workspace_bytes()  # capacity of tq_decode_attention_static's scratch


def tq_decode_attention_static(k_ctx, v_ctx, q, k_cache, v_cache, out, B, Hq, Hkv, L, seq_lens=None,
                               scale=0.0, stream=None):
    """tq_decode_attention with its scratch in the library's static device area (no workspace
    argument, no allocation); calls that overlap on one device race on that area."""
    qp, qd = _q_args(q)
    _check(lib.tq_decode_attention_static(k_ctx.handle, v_ctx.handle, qp, qd, _ptr(k_cache), _ptr(v_cache),
                                          _ptr(seq_lens), B, Hq, Hkv, L, scale, _ptr(out), _stream(stream)),
           "tq_decode_attention_static")


def tq_decode_partial_merge(k_ctx, v_ctx, k_cache, v_cache, out, workspace, B, Hq, Hkv, L, seq_lens=None,
                            stream=None):
    _check(lib.tq_decode_partial_merge(k_ctx.handle, v_ctx.handle, _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                       B, Hq, Hkv, L, _ptr(out), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)),
           "tq_decode_partial_merge")


def tq_decode_prepare_q(k_ctx, v_ctx, q, workspace, B, Hq, Hkv, L, scale=0.0, stream=None):
    qp, qd = _q_args(q)
    _check(lib.tq_decode_prepare_q(k_ctx.handle, v_ctx.handle, qp, qd, B, Hq, Hkv, L, scale, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "tq_decode_prepare_q")


def tq_decode_partial(k_ctx, v_ctx, k_cache, v_cache, workspace, B, Hq, Hkv, L, seq_lens=None, scores=None,
                      stream=None):
    _check(lib.tq_decode_partial(k_ctx.handle, v_ctx.handle, _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens),
                                 B, Hq, Hkv, L, _ptr(scores), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)),
           "tq_decode_partial")


def tq_decode_combine(k_ctx, v_ctx, out, workspace, B, Hq, Hkv, L, stream=None):
    _check(lib.tq_decode_combine(k_ctx.handle, v_ctx.handle, B, Hq, Hkv, L, _ptr(out), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)),
           "tq_decode_combine")


def alloc_workspace(nbytes, device="cuda"):
    """A 256-byte aligned uint8 CUDA tensor of at least ``nbytes`` bytes."""
    import torch
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def alloc_cache(fmt, n_rows, device="cuda", d=D):
    """A uint8 CUDA tensor sized by tq_cache_bytes (readable to the next 16-byte boundary);
    rows of head dimension 256 take two 128-element blocks each."""
    import torch
    return torch.zeros(tq_cache_bytes(fmt, n_rows * d // D), dtype=torch.uint8, device=device)
