// The extern "C" entry points of tq.h: argument validation on the host, context
// construction, and dispatch to the kernel launchers.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "tq_internal.h"

namespace tq {
const char *last_error();
}

using namespace tq;

namespace {

tq_status fail(tq_status s, const char *msg) {
  set_error("%s", msg);
  return s;
}

tq_status cuda_fail(cudaError_t e, const char *where) {
  set_error("%s: %s", where, cudaGetErrorString(e));
  (void)cudaGetLastError();  // a reported failure does not surface again in a later launch check
  return TQ_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

int code_bits(int fmt) {
  switch (fmt) {
    case TQ_FMT_TURBO4: return 4;
    case TQ_FMT_TURBO3: return 3;
    case TQ_FMT_PROD3: return 2;
    default: return 0;
  }
}

// The d x d rotation R (row-major fp32) and, for the WHT, its sign bits (d / 32 words).
tq_status build_rotation(int kind, int d, uint64_t seed, std::vector<float> &r, uint32_t *neg) {
  r.assign((size_t)d * d, 0.f);
  if (kind == TQ_ROT_DENSE) {
    std::vector<double> pi((size_t)d * d);
    if (!dense_rotation_f64(seed, d, pi.data())) return fail(TQ_ERR_INVALID_ARG, "rank-deficient Gaussian");
    for (size_t i = 0; i < pi.size(); ++i) r[i] = (float)pi[i];
    return TQ_OK;
  }
  std::vector<uint64_t> out(d);
  splitmix64_fill(seed, out.data(), d);
  for (int i = 0; i < d / 32; ++i) neg[i] = 0;
  std::vector<double> s(d);
  for (int j = 0; j < d; ++j) {
    const bool minus = (out[j] >> 63) != 0;
    s[j] = minus ? -1.0 : 1.0;
    if (minus) neg[j / 32] |= 1u << (j % 32);
  }
  // R = (1/sqrt(d)) H D with H the Sylvester Hadamard matrix, H[i][j] = (-1)^popcount(i & j).
  const double inv = 1.0 / std::sqrt((double)d);
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) {
      const double h = (__builtin_popcount(i & j) & 1) ? -1.0 : 1.0;
      r[(size_t)i * d + j] = (float)(h * s[j] * inv);
    }
  return TQ_OK;
}

template <typename T>
tq_status to_device(T **dst, const T *src, size_t n) {
  cudaError_t e = cudaMalloc((void **)dst, n * sizeof(T));
  if (e != cudaSuccess) return fail(TQ_ERR_ALLOC, "cudaMalloc failed");
  e = cudaMemcpy(*dst, src, n * sizeof(T), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
  return TQ_OK;
}


tq_status check_decode_common(const tq_ctx *k, const tq_ctx *v, int B, int Hq, int Hkv, int L,
                              DecodeShape *shape) {
  if (!k || !v) return fail(TQ_ERR_INVALID_ARG, "null context");
  if (k->device != v->device) return fail(TQ_ERR_INVALID_ARG, "the key and value contexts belong to different devices");
  tq_status st = check_current_device(k->device, "decode");
  if (st != TQ_OK) return st;
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1) return fail(TQ_ERR_INVALID_ARG, "B, Hq, Hkv and L must be >= 1");
  if (Hq % Hkv != 0) return fail(TQ_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
  if (!decode_pair_supported(k, v))
    return fail(TQ_ERR_UNSUPPORTED, "no decode kernel for this (key, value) format pair");
  if (!decode_shape(k, v, B, Hq, Hkv, L, shape)) return fail(TQ_ERR_UNSUPPORTED, "shape too large");
  return TQ_OK;
}

// Head dimension 256: turbo4 keys and values only, through the kernels of tq_d256.cu.
bool is_d256(const tq_ctx *k, const tq_ctx *v) { return (k && k->d == D256) || (v && v->d == D256); }

tq_status check_d256(const tq_ctx *k, const tq_ctx *v, int B, int Hq, int Hkv, int L, D256Shape *s) {
  if (!k || !v) return fail(TQ_ERR_INVALID_ARG, "null context");
  if (k->device != v->device) return fail(TQ_ERR_INVALID_ARG, "the key and value contexts belong to different devices");
  tq_status st = check_current_device(k->device, "decode");
  if (st != TQ_OK) return st;
  if (k->d != D256 || v->d != D256 || k->fmt != TQ_FMT_TURBO4 || v->fmt != TQ_FMT_TURBO4)
    return fail(TQ_ERR_UNSUPPORTED, "at head dimension 256 both contexts must be TURBO4 with d = 256");
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1) return fail(TQ_ERR_INVALID_ARG, "B, Hq, Hkv and L must be >= 1");
  if (Hq % Hkv != 0) return fail(TQ_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
  if (!d256_shape(k, B, Hq, Hkv, L, s)) return fail(TQ_ERR_UNSUPPORTED, "shape too large");
  return TQ_OK;
}

tq_status check_workspace256(const D256Shape &s, void *ws, size_t bytes, Workspace *w) {
  if (!ws) return fail(TQ_ERR_INVALID_ARG, "null workspace");
  if (!aligned(ws, 256)) return fail(TQ_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (bytes < d256_workspace(s, ws, w)) return fail(TQ_ERR_WORKSPACE, "workspace smaller than tq_decode_workspace_size()");
  return TQ_OK;
}

tq_status check_q(const void *q, int q_dtype, float scale) {
  if (!q) return fail(TQ_ERR_INVALID_ARG, "null q");
  if (q_dtype != TQ_DTYPE_F32 && q_dtype != TQ_DTYPE_BF16 && q_dtype != TQ_DTYPE_F16)
    return fail(TQ_ERR_INVALID_ARG, "bad q dtype");
  if (!aligned(q, 16)) return fail(TQ_ERR_ALIGNMENT, "q must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(TQ_ERR_INVALID_ARG, "scale must be finite");
  return TQ_OK;
}

tq_status check_caches(const void *k_cache, const void *v_cache, const int32_t *seq_lens) {
  if (!k_cache || !v_cache) return fail(TQ_ERR_INVALID_ARG, "null cache");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return fail(TQ_ERR_ALIGNMENT, "caches must be 16-byte aligned");
  if (seq_lens && !aligned(seq_lens, 4)) return fail(TQ_ERR_ALIGNMENT, "seq_lens must be 4-byte aligned");
  return TQ_OK;
}

// The d = 256 decode stages: q preparation, split-K partials, combine (mask: 1, 2, 4).
tq_status run_d256(const tq_ctx *k, const tq_ctx *v, const void *q, int q_dtype, const void *kc, const void *vc,
                   const int32_t *seq_lens, const D256Shape &s, float scale, float *out, const Workspace &w,
                   cudaStream_t st, int stages) {
  cudaError_t e = cudaSuccess;
  if ((stages & 1) && (e = launch_prepare_q256(k, q, q_dtype, s, scale == 0.f ? 1.0f / 16.0f : scale, w, st)) !=
                          cudaSuccess)
    return cuda_fail(e, "prepare_q launch");
  if ((stages & 2) && (e = launch_partial_d256(k, v, (const uint8_t *)kc, (const uint8_t *)vc, seq_lens, s, w, st)) !=
                          cudaSuccess)
    return cuda_fail(e, "partial launch");
  if ((stages & 4) && (e = launch_combine_d256(v, s, out, w, st)) != cudaSuccess) return cuda_fail(e, "combine launch");
  return TQ_OK;
}

tq_status check_workspace(const DecodeShape &s, void *ws, size_t bytes, Workspace *w) {
  if (!ws) return fail(TQ_ERR_INVALID_ARG, "null workspace");
  if (!aligned(ws, 256)) return fail(TQ_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  *w = carve_workspace(s, ws);
  if (bytes < w->bytes) return fail(TQ_ERR_WORKSPACE, "workspace smaller than tq_decode_workspace_size()");
  return TQ_OK;
}

}  // namespace

namespace tq {
tq_status check_current_device(int device, const char *who) {
  int cur = -1;
  const cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) {
    set_error("%s: cannot read the current device: %s", who, cudaGetErrorString(e));
    return TQ_ERR_CUDA;
  }
  if (cur != device) {
    set_error("%s: the context belongs to device %d but device %d is current", who, device, cur);
    return TQ_ERR_INVALID_ARG;
  }
  return TQ_OK;
}

bool decode_pair_supported(const tq_ctx *k, const tq_ctx *v) {
  if (k->d != D || v->d != D) return false;  // d = 256 has its own path (turbo4 only)
  return ((k->fmt == TQ_FMT_TURBO4 || k->fmt == TQ_FMT_TURBO3) &&
          (v->fmt == TQ_FMT_TURBO4 || v->fmt == TQ_FMT_TURBO3)) ||
         (k->fmt == TQ_FMT_PROD3 && v->fmt == TQ_FMT_VGROUP2);
}
}  // namespace tq

extern "C" {

const char *tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported";
    case TQ_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case TQ_ERR_CUDA: return "CUDA error";
    case TQ_ERR_ALLOC: return "allocation failed";
    case TQ_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

const char *tq_last_error(void) { return tq::last_error(); }

int64_t tq_row_bytes(int format) {
  switch (format) {
    case TQ_FMT_TURBO4: return 68;
    case TQ_FMT_TURBO3: return 56;
    case TQ_FMT_PROD3: return 56;
    case TQ_FMT_VGROUP2: return 48;
  }
  return -1;
}

size_t tq_cache_bytes(int format, int64_t n_rows) {
  const int64_t rb = tq_row_bytes(format);
  if (rb < 0 || n_rows < 0) return 0;
  return ((size_t)n_rows * (size_t)rb + 15) & ~(size_t)15;
}

tq_status tq_make_codebook(int bits, int d, int kind, float *centroids, float *boundaries) {
  if (d != D && d != D256) return fail(TQ_ERR_UNSUPPORTED, "d must be 128 or 256");
  if (bits < 1 || bits > 4) return fail(TQ_ERR_UNSUPPORTED, "bits must be 1..4");
  if (kind != TQ_CB_QUANTILE && kind != TQ_CB_LLOYD && kind != TQ_CB_SPHERE)
    return fail(TQ_ERR_INVALID_ARG, "bad codebook kind");
  if (!centroids) return fail(TQ_ERR_INVALID_ARG, "null centroids");
  double c[16];
  if (!make_codebook_f64(bits, d, kind, c)) return fail(TQ_ERR_INVALID_ARG, "codebook construction failed");
  store_codebook(c, 1 << bits, centroids, boundaries);
  return TQ_OK;
}

tq_status tq_make_rotation(int kind, int d, uint64_t seed, float *out) {
  if (d != D && d != D256) return fail(TQ_ERR_UNSUPPORTED, "d must be 128 or 256");
  if (!out) return fail(TQ_ERR_INVALID_ARG, "null output");
  if (kind != TQ_ROT_WHT && kind != TQ_ROT_DENSE) return fail(TQ_ERR_INVALID_ARG, "bad rotation kind");
  std::vector<float> r;
  uint32_t neg[8];
  tq_status s = build_rotation(kind, d, seed, r, neg);
  if (s != TQ_OK) return s;
  if (kind == TQ_ROT_DENSE) {
    std::memcpy(out, r.data(), r.size() * sizeof(float));
  } else {
    for (int j = 0; j < d; ++j) out[j] = ((neg[j / 32] >> (j % 32)) & 1u) ? -1.f : 1.f;
  }
  return TQ_OK;
}

tq_status tq_make_qjl_matrix(int d, uint64_t seed, float *out) {
  if (d != D) return fail(TQ_ERR_UNSUPPORTED, "only d = 128 is supported");
  if (!out) return fail(TQ_ERR_INVALID_ARG, "null output");
  std::vector<double> g((size_t)D * D);
  gaussian_fill(seed, g.data(), g.size());
  for (size_t i = 0; i < g.size(); ++i) out[i] = (float)g[i];
  return TQ_OK;
}

tq_status tq_ctx_create(const tq_params *params, tq_ctx **out) {
  if (!params || !out) return fail(TQ_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  const tq_params &p = *params;
  if (p.format < TQ_FMT_TURBO4 || p.format > TQ_FMT_VGROUP2) return fail(TQ_ERR_INVALID_ARG, "bad format");
  if (p.d != D && !(p.d == D256 && p.format == TQ_FMT_TURBO4))
    return fail(TQ_ERR_UNSUPPORTED, "d = 128 for every format, d = 256 for TURBO4");
  const bool rotated = p.format != TQ_FMT_VGROUP2;
  if (rotated && p.rotation != TQ_ROT_WHT && p.rotation != TQ_ROT_DENSE)
    return fail(TQ_ERR_INVALID_ARG, "bad rotation kind");
  if (rotated && p.codebook != TQ_CB_DEFAULT && p.codebook != TQ_CB_QUANTILE && p.codebook != TQ_CB_LLOYD &&
      p.codebook != TQ_CB_SPHERE)
    return fail(TQ_ERR_INVALID_ARG, "bad codebook kind");
  if (p.format == TQ_FMT_PROD3 && p.qjl_seed == p.rot_seed)
    return fail(TQ_ERR_INVALID_ARG, "the QJL seed must differ from the rotation seed");
  if ((p.qjl_shrink != 0 && p.qjl_shrink != 1) || p.reserved != 0)
    return fail(TQ_ERR_INVALID_ARG, "qjl_shrink must be 0 or 1 and reserved 0");

  tq_ctx *c = new (std::nothrow) tq_ctx();
  if (!c) return fail(TQ_ERR_ALLOC, "host allocation failed");
  c->p = p;
  c->fmt = p.format;
  c->d = p.d;
  const int d = p.d;
  c->qjl_factor = (p.format == TQ_FMT_PROD3 && p.qjl_shrink) ? (float)(2.0 / 3.14159265358979323846) : 1.0f;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&c->reserved_smem, cudaDevAttrReservedSharedMemoryPerBlock, c->device);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "cudaGetDevice");
  }
  tq_status s = TQ_OK;
  if (rotated) {
    const int bits = code_bits(p.format);
    int kind = p.codebook;
    if (kind == TQ_CB_DEFAULT) kind = (p.format == TQ_FMT_TURBO4) ? TQ_CB_QUANTILE : TQ_CB_LLOYD;
    double c64[16];
    make_codebook_f64(bits, d, kind, c64);
    c->cb.bits = bits;
    c->cb.K = 1 << bits;
    store_codebook(c64, c->cb.K, c->cb.c, c->cb.b);
    c->f16 = make_f16_table(c->cb.c, c->cb.K);
    c->bt = make_bucket_table(c->cb.b, c->cb.K - 1);
    std::vector<float> r;
    s = build_rotation(p.rotation, d, p.rot_seed, r, c->wht_neg);
    if (s == TQ_OK) s = to_device(&c->d_pi, r.data(), r.size());
    if (s == TQ_OK) {
      std::vector<float> rt((size_t)d * d);
      for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) rt[(size_t)j * d + i] = r[(size_t)i * d + j];
      s = to_device(&c->d_pit, rt.data(), rt.size());
    }
    if (s == TQ_OK && p.rotation == TQ_ROT_DENSE && d == D) {
      // bf16 hi + lo parts of R for the tensor-core write: hi = RN(r), lo = RN(r - hi)
      std::vector<uint16_t> rb(2 * (size_t)D * D);
      for (size_t i = 0; i < (size_t)D * D; ++i) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(r[i]);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r[i] - __bfloat162float(hi));
        rb[i] = __bfloat16_as_ushort(hi);
        rb[(size_t)D * D + i] = __bfloat16_as_ushort(lo);
      }
      s = to_device(&c->d_pib, rb.data(), rb.size());
    }
    if (s == TQ_OK && p.format == TQ_FMT_PROD3) {
      std::vector<float> S((size_t)D * D), St((size_t)D * D);
      tq_make_qjl_matrix(D, p.qjl_seed, S.data());
      for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) St[(size_t)j * D + i] = S[(size_t)i * D + j];
      s = to_device(&c->d_S, S.data(), S.size());
      if (s == TQ_OK) s = to_device(&c->d_St, St.data(), St.size());
    }
  }
  if (s == TQ_OK && rotated) s = to_device(&c->d_bt, &c->bt, 1);
  if (s == TQ_OK) {
    e = cudaMalloc((void **)&c->d_status, sizeof(int32_t));
    if (e != cudaSuccess) s = fail(TQ_ERR_ALLOC, "cudaMalloc failed");
    else if ((e = cudaMemset(c->d_status, 0, sizeof(int32_t))) != cudaSuccess) s = cuda_fail(e, "cudaMemset");
  }
  if (s != TQ_OK) {
    tq_ctx_destroy(c);
    return s;
  }
  *out = c;
  return TQ_OK;
}

tq_status tq_ctx_destroy(tq_ctx *ctx) {
  if (!ctx) return TQ_OK;
  cudaFree(ctx->d_pi);
  cudaFree(ctx->d_pit);
  cudaFree(ctx->d_S);
  cudaFree(ctx->d_St);
  cudaFree(ctx->d_pib);
  cudaFree(ctx->d_bt);
  cudaFree(ctx->d_status);
  delete ctx;
  return TQ_OK;
}

tq_status tq_ctx_device_status(const tq_ctx *ctx, int32_t *status, int clear) {
  if (!ctx || !status) return fail(TQ_ERR_INVALID_ARG, "null argument");
  tq_status st = check_current_device(ctx->device, "tq_ctx_device_status");
  if (st != TQ_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  e = cudaMemcpy(status, ctx->d_status, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
  if (clear && (e = cudaMemset(ctx->d_status, 0, sizeof(int32_t))) != cudaSuccess) return cuda_fail(e, "cudaMemset");
  return TQ_OK;
}

namespace {
// The argument checks of tq_quantize_set_rows for a call with n_rows >= 1.
tq_status check_write_args(const void *src, int src_dtype, int64_t src_row_stride, const int64_t *row_ids,
                           const void *dst_cache, int64_t n_rows, int64_t dst_rows, int d = D) {
  if (!src || !dst_cache) return fail(TQ_ERR_INVALID_ARG, "null source or cache");
  if (src_dtype != TQ_DTYPE_F32 && src_dtype != TQ_DTYPE_BF16)
    return fail(TQ_ERR_UNSUPPORTED, "source dtype must be F32 or BF16");
  if (src_row_stride < d) return fail(TQ_ERR_INVALID_ARG, "source row stride below the head dimension");
  if (dst_rows < 1) return fail(TQ_ERR_INVALID_ARG, "dst_rows < 1");
  if (!row_ids && dst_rows < n_rows) return fail(TQ_ERR_INVALID_ARG, "identity slots need dst_rows >= n_rows");
  const size_t esz = src_dtype == TQ_DTYPE_F32 ? 4 : 2;
  const size_t need = src_dtype == TQ_DTYPE_F32 ? 16 : 8;
  if (!aligned(src, need) || ((size_t)src_row_stride * esz) % need != 0)
    return fail(TQ_ERR_ALIGNMENT, "source rows must be 16-byte (F32) or 8-byte (BF16) aligned");
  if (!aligned(dst_cache, 16)) return fail(TQ_ERR_ALIGNMENT, "cache must be 16-byte aligned");
  if (row_ids && !aligned(row_ids, 8)) return fail(TQ_ERR_ALIGNMENT, "row_ids must be 8-byte aligned");
  return TQ_OK;
}
}  // namespace

tq_status tq_quantize_set_rows(const tq_ctx *ctx, const void *src, int src_dtype, int64_t n_rows,
                               int64_t src_row_stride, const int64_t *row_ids, void *dst_cache,
                               int64_t dst_rows, tq_stream_t stream) {
  if (!ctx) return fail(TQ_ERR_INVALID_ARG, "null context");
  if (n_rows < 0) return fail(TQ_ERR_INVALID_ARG, "n_rows < 0");
  if (n_rows == 0) return TQ_OK;
  tq_status st = check_current_device(ctx->device, "tq_quantize_set_rows");
  if (st != TQ_OK) return st;
  if ((st = check_write_args(src, src_dtype, src_row_stride, row_ids, dst_cache, n_rows, dst_rows, ctx->d)) !=
      TQ_OK)
    return st;
  WriteLaunch w{src, src_dtype, n_rows, src_row_stride, row_ids, (uint8_t *)dst_cache, dst_rows};
  cudaError_t e = ctx->d == D256 ? launch_write_d256(ctx, w, (cudaStream_t)stream)
                                 : launch_write(ctx, w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "write kernel launch");
  return TQ_OK;
}

tq_status tq_dequantize(const tq_ctx *ctx, const void *cache, int64_t n_rows, int unrotate,
                        float *dst, tq_stream_t stream) {
  if (!ctx) return fail(TQ_ERR_INVALID_ARG, "null context");
  if (n_rows < 0) return fail(TQ_ERR_INVALID_ARG, "n_rows < 0");
  if (n_rows == 0) return TQ_OK;
  tq_status st = check_current_device(ctx->device, "tq_dequantize");
  if (st != TQ_OK) return st;
  if (!cache || !dst) return fail(TQ_ERR_INVALID_ARG, "null cache or output");
  if (!aligned(cache, 16)) return fail(TQ_ERR_ALIGNMENT, "cache must be 16-byte aligned");
  if (!aligned(dst, 4)) return fail(TQ_ERR_ALIGNMENT, "output must be 4-byte aligned");
  cudaError_t e = ctx->d == D256 ? launch_dequant_d256(ctx, (const uint8_t *)cache, n_rows, unrotate, dst,
                                                      (cudaStream_t)stream)
                                 : launch_dequantize(ctx, (const uint8_t *)cache, n_rows, unrotate, dst,
                                                     (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequantize launch");
  return TQ_OK;
}

tq_status tq_decode_num_splits(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int Hq, int Hkv,
                               int L, int *n_split) {
  if (is_d256(k_ctx, v_ctx)) {
    if (!n_split) return fail(TQ_ERR_INVALID_ARG, "null output");
    D256Shape s;
    tq_status st = check_d256(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
    if (st == TQ_OK) *n_split = s.n_split;
    return st;
  }
  if (!n_split) return fail(TQ_ERR_INVALID_ARG, "null output");
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  *n_split = s.n_part;
  return TQ_OK;
}

tq_status tq_decode_workspace_size(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int Hq,
                                   int Hkv, int L, size_t *bytes) {
  if (is_d256(k_ctx, v_ctx)) {
    if (!bytes) return fail(TQ_ERR_INVALID_ARG, "null output");
    D256Shape s;
    tq_status st = check_d256(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
    if (st == TQ_OK) *bytes = d256_workspace(s, nullptr, nullptr);
    return st;
  }
  if (!bytes) return fail(TQ_ERR_INVALID_ARG, "null output");
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  *bytes = carve_workspace(s, nullptr).bytes;
  return TQ_OK;
}

tq_status tq_decode_prepare_q(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *q,
                              int q_dtype, int B, int Hq, int Hkv, int L, float scale,
                              void *workspace, size_t workspace_bytes, tq_stream_t stream) {
  if (is_d256(k_ctx, v_ctx)) {
    D256Shape s;
    Workspace w;
    tq_status st = check_d256(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
    if (st == TQ_OK) st = check_q(q, q_dtype, scale);
    if (st == TQ_OK) st = check_workspace256(s, workspace, workspace_bytes, &w);
    if (st != TQ_OK) return st;
    return run_d256(k_ctx, v_ctx, q, q_dtype, nullptr, nullptr, nullptr, s, scale, nullptr, w, (cudaStream_t)stream, 1);
  }
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (!q) return fail(TQ_ERR_INVALID_ARG, "null q");
  if (q_dtype != TQ_DTYPE_F32 && q_dtype != TQ_DTYPE_BF16 && q_dtype != TQ_DTYPE_F16)
    return fail(TQ_ERR_INVALID_ARG, "bad q dtype");
  if (!aligned(q, 16)) return fail(TQ_ERR_ALIGNMENT, "q must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(TQ_ERR_INVALID_ARG, "scale must be finite");
  if (scale == 0.f) scale = 1.0f / std::sqrt((float)D);
  Workspace w;
  if ((st = check_workspace(s, workspace, workspace_bytes, &w)) != TQ_OK) return st;
  cudaError_t e = launch_prepare_q(k_ctx, q, q_dtype, s, scale, w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "prepare_q launch");
  return TQ_OK;
}

tq_status tq_decode_partial(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *k_cache,
                            const void *v_cache, const int32_t *seq_lens, int B, int Hq, int Hkv,
                            int L, float *scores_dbg, void *workspace, size_t workspace_bytes,
                            tq_stream_t stream) {
  if (is_d256(k_ctx, v_ctx)) {
    D256Shape s;
    Workspace w;
    tq_status st = check_d256(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
    if (st == TQ_OK) st = check_caches(k_cache, v_cache, seq_lens);
    if (st == TQ_OK && scores_dbg) st = fail(TQ_ERR_UNSUPPORTED, "no score output at head dimension 256");
    if (st == TQ_OK) st = check_workspace256(s, workspace, workspace_bytes, &w);
    if (st != TQ_OK) return st;
    return run_d256(k_ctx, v_ctx, nullptr, 0, k_cache, v_cache, seq_lens, s, 0.f, nullptr, w, (cudaStream_t)stream, 2);
  }
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (!k_cache || !v_cache) return fail(TQ_ERR_INVALID_ARG, "null cache");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return fail(TQ_ERR_ALIGNMENT, "caches must be 16-byte aligned");
  if (seq_lens && !aligned(seq_lens, 4)) return fail(TQ_ERR_ALIGNMENT, "seq_lens must be 4-byte aligned");
  if (scores_dbg && !aligned(scores_dbg, 4)) return fail(TQ_ERR_ALIGNMENT, "scores must be 4-byte aligned");
  Workspace w;
  if ((st = check_workspace(s, workspace, workspace_bytes, &w)) != TQ_OK) return st;
  cudaError_t e = launch_partial(k_ctx, v_ctx, (const uint8_t *)k_cache, (const uint8_t *)v_cache,
                                 seq_lens, s, scores_dbg, w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "partial launch");
  return TQ_OK;
}

tq_status tq_decode_combine(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int Hq, int Hkv,
                            int L, float *out, void *workspace, size_t workspace_bytes,
                            tq_stream_t stream) {
  if (is_d256(k_ctx, v_ctx)) {
    D256Shape s;
    Workspace w;
    tq_status st = check_d256(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
    if (st == TQ_OK && !out) st = fail(TQ_ERR_INVALID_ARG, "null output");
    if (st == TQ_OK && !aligned(out, 16)) st = fail(TQ_ERR_ALIGNMENT, "output must be 16-byte aligned at d = 256");
    if (st == TQ_OK) st = check_workspace256(s, workspace, workspace_bytes, &w);
    if (st != TQ_OK) return st;
    return run_d256(k_ctx, v_ctx, nullptr, 0, nullptr, nullptr, nullptr, s, 0.f, out, w, (cudaStream_t)stream, 4);
  }
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (!out) return fail(TQ_ERR_INVALID_ARG, "null output");
  if (!aligned(out, 4)) return fail(TQ_ERR_ALIGNMENT, "output must be 4-byte aligned");
  Workspace w;
  if ((st = check_workspace(s, workspace, workspace_bytes, &w)) != TQ_OK) return st;
  cudaError_t e = launch_combine(k_ctx, v_ctx, s, out, w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return TQ_OK;
}

tq_status tq_decode_partial_merge(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *k_cache,
                                  const void *v_cache, const int32_t *seq_lens, int B, int Hq, int Hkv,
                                  int L, float *out, void *workspace, size_t workspace_bytes,
                                  tq_stream_t stream) {
  if (is_d256(k_ctx, v_ctx)) {
    D256Shape s;
    Workspace w;
    tq_status st = check_d256(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
    if (st == TQ_OK) st = check_caches(k_cache, v_cache, seq_lens);
    if (st == TQ_OK && !out) st = fail(TQ_ERR_INVALID_ARG, "null output");
    if (st == TQ_OK && !aligned(out, 16)) st = fail(TQ_ERR_ALIGNMENT, "output must be 16-byte aligned at d = 256");
    if (st == TQ_OK) st = check_workspace256(s, workspace, workspace_bytes, &w);
    if (st != TQ_OK) return st;
    return run_d256(k_ctx, v_ctx, nullptr, 0, k_cache, v_cache, seq_lens, s, 0.f, out, w, (cudaStream_t)stream, 6);
  }
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (!k_cache || !v_cache) return fail(TQ_ERR_INVALID_ARG, "null cache");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return fail(TQ_ERR_ALIGNMENT, "caches must be 16-byte aligned");
  if (seq_lens && !aligned(seq_lens, 4)) return fail(TQ_ERR_ALIGNMENT, "seq_lens must be 4-byte aligned");
  if (!out) return fail(TQ_ERR_INVALID_ARG, "null output");
  if (!aligned(out, 4)) return fail(TQ_ERR_ALIGNMENT, "output must be 4-byte aligned");
  Workspace w;
  if ((st = check_workspace(s, workspace, workspace_bytes, &w)) != TQ_OK) return st;
  bool fused = false;
  cudaError_t e = launch_partial(k_ctx, v_ctx, (const uint8_t *)k_cache, (const uint8_t *)v_cache, seq_lens,
                                 s, nullptr, w, (cudaStream_t)stream, false, out, &fused);
  if (e != cudaSuccess) return cuda_fail(e, "partial launch");
  if (fused) return TQ_OK;
  e = launch_combine(k_ctx, v_ctx, s, out, w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return TQ_OK;
}

tq_status tq_decode_num_launches(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int Hq, int Hkv,
                                 int L, int *n) {
  if (is_d256(k_ctx, v_ctx)) {
    if (!n) return fail(TQ_ERR_INVALID_ARG, "null output");
    D256Shape s;
    tq_status st = check_d256(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
    if (st == TQ_OK) *n = 3;
    return st;
  }
  if (!n) return fail(TQ_ERR_INVALID_ARG, "null output");
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  *n = partial_fuses_combine(s) ? 2 : 3;
  return TQ_OK;
}

tq_status tq_decode_attention(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *q,
                              int q_dtype, const void *k_cache, const void *v_cache,
                              const int32_t *seq_lens, int B, int Hq, int Hkv, int L, float scale,
                              float *out, float *scores_dbg, void *workspace,
                              size_t workspace_bytes, tq_stream_t stream) {
  if (is_d256(k_ctx, v_ctx)) {
    D256Shape s;
    Workspace w;
    tq_status st = check_d256(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
    if (st == TQ_OK) st = check_caches(k_cache, v_cache, seq_lens);
    if (st == TQ_OK && scores_dbg) st = fail(TQ_ERR_UNSUPPORTED, "no score output at head dimension 256");
    if (st == TQ_OK && !out) st = fail(TQ_ERR_INVALID_ARG, "null output");
    if (st == TQ_OK && !aligned(out, 16)) st = fail(TQ_ERR_ALIGNMENT, "output must be 16-byte aligned at d = 256");
    if (st == TQ_OK) st = check_q(q, q_dtype, scale);
    if (st == TQ_OK) st = check_workspace256(s, workspace, workspace_bytes, &w);
    if (st != TQ_OK) return st;
    return run_d256(k_ctx, v_ctx, q, q_dtype, k_cache, v_cache, seq_lens, s, scale, out, w, (cudaStream_t)stream, 7);
  }
  // the three stages' checks up front, so nothing is launched for a call that fails
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (!k_cache || !v_cache) return fail(TQ_ERR_INVALID_ARG, "null cache");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return fail(TQ_ERR_ALIGNMENT, "caches must be 16-byte aligned");
  if (seq_lens && !aligned(seq_lens, 4)) return fail(TQ_ERR_ALIGNMENT, "seq_lens must be 4-byte aligned");
  if (scores_dbg && !aligned(scores_dbg, 4)) return fail(TQ_ERR_ALIGNMENT, "scores must be 4-byte aligned");
  if (!out) return fail(TQ_ERR_INVALID_ARG, "null output");
  if (!aligned(out, 4)) return fail(TQ_ERR_ALIGNMENT, "output must be 4-byte aligned");
  st = tq_decode_prepare_q(k_ctx, v_ctx, q, q_dtype, B, Hq, Hkv, L, scale, workspace,
                           workspace_bytes, stream);
  if (st != TQ_OK) return st;
  Workspace w;
  if ((st = check_workspace(s, workspace, workspace_bytes, &w)) != TQ_OK) return st;
  // the split-K kernel merges the splits itself when it can (the CTA completing a unit
  // writes its outputs); otherwise the combine kernel does
  bool fused = false;
  cudaError_t e = launch_partial(k_ctx, v_ctx, (const uint8_t *)k_cache, (const uint8_t *)v_cache, seq_lens,
                                 s, scores_dbg, w, (cudaStream_t)stream, false, out, &fused);
  if (e != cudaSuccess) return cuda_fail(e, "partial launch");
  if (fused) return TQ_OK;
  e = launch_combine(k_ctx, v_ctx, s, out, w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return TQ_OK;
}


tq_status tq_decode_step(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *new_k, const void *new_v,
                         int src_dtype, int64_t n_rows, int64_t src_row_stride, const int64_t *row_ids,
                         const void *q, int q_dtype, void *k_cache, void *v_cache,
                         const int32_t *seq_lens, int B, int Hq, int Hkv, int L, float scale, float *out,
                         void *workspace, size_t workspace_bytes, tq_stream_t stream) {
  if (is_d256(k_ctx, v_ctx)) {
    D256Shape s;
    Workspace w;
    tq_status st = check_d256(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
    if (st != TQ_OK) return st;
    if (n_rows < 0) return fail(TQ_ERR_INVALID_ARG, "n_rows < 0");
    const int64_t dst_rows = (int64_t)B * Hkv * L;
    if (n_rows > 0 &&
        ((st = check_write_args(new_k, src_dtype, src_row_stride, row_ids, k_cache, n_rows, dst_rows, D256)) != TQ_OK ||
         (st = check_write_args(new_v, src_dtype, src_row_stride, row_ids, v_cache, n_rows, dst_rows, D256)) != TQ_OK))
      return st;
    if ((st = check_caches(k_cache, v_cache, seq_lens)) != TQ_OK || (st = check_q(q, q_dtype, scale)) != TQ_OK)
      return st;
    if (!out) return fail(TQ_ERR_INVALID_ARG, "null output");
    if (!aligned(out, 16)) return fail(TQ_ERR_ALIGNMENT, "output must be 16-byte aligned at d = 256");
    if ((st = check_workspace256(s, workspace, workspace_bytes, &w)) != TQ_OK) return st;
    const cudaStream_t cs = (cudaStream_t)stream;
    if (n_rows > 0) {
      const WriteLaunch wk{new_k, src_dtype, n_rows, src_row_stride, row_ids, (uint8_t *)k_cache, dst_rows};
      const WriteLaunch wv{new_v, src_dtype, n_rows, src_row_stride, row_ids, (uint8_t *)v_cache, dst_rows};
      cudaError_t e;
      if ((e = launch_write_d256(k_ctx, wk, cs)) != cudaSuccess || (e = launch_write_d256(v_ctx, wv, cs)) != cudaSuccess)
        return cuda_fail(e, "write kernel launch");
    }
    return run_d256(k_ctx, v_ctx, q, q_dtype, k_cache, v_cache, seq_lens, s, scale, out, w, cs, 7);
  }
  // every check of the three calls first, so that nothing is launched for a call that fails
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (n_rows < 0) return fail(TQ_ERR_INVALID_ARG, "n_rows < 0");
  const int64_t dst_rows = (int64_t)B * Hkv * L;
  if (n_rows > 0) {
    if ((st = check_write_args(new_k, src_dtype, src_row_stride, row_ids, k_cache, n_rows, dst_rows)) != TQ_OK ||
        (st = check_write_args(new_v, src_dtype, src_row_stride, row_ids, v_cache, n_rows, dst_rows)) != TQ_OK)
      return st;
  }
  if (!k_cache || !v_cache) return fail(TQ_ERR_INVALID_ARG, "null cache");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return fail(TQ_ERR_ALIGNMENT, "caches must be 16-byte aligned");
  if (!q) return fail(TQ_ERR_INVALID_ARG, "null q");
  if (q_dtype != TQ_DTYPE_F32 && q_dtype != TQ_DTYPE_BF16 && q_dtype != TQ_DTYPE_F16)
    return fail(TQ_ERR_INVALID_ARG, "bad q dtype");
  if (!aligned(q, 16)) return fail(TQ_ERR_ALIGNMENT, "q must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(TQ_ERR_INVALID_ARG, "scale must be finite");
  if (seq_lens && !aligned(seq_lens, 4)) return fail(TQ_ERR_ALIGNMENT, "seq_lens must be 4-byte aligned");
  if (!out) return fail(TQ_ERR_INVALID_ARG, "null output");
  if (!aligned(out, 4)) return fail(TQ_ERR_ALIGNMENT, "output must be 4-byte aligned");
  Workspace w;
  if ((st = check_workspace(s, workspace, workspace_bytes, &w)) != TQ_OK) return st;
  if (scale == 0.f) scale = 1.0f / std::sqrt((float)D);

  const WriteLaunch wk{new_k, src_dtype, n_rows, src_row_stride, row_ids, (uint8_t *)k_cache, dst_rows};
  const WriteLaunch wv{new_v, src_dtype, n_rows, src_row_stride, row_ids, (uint8_t *)v_cache, dst_rows};
  const cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e;
  if (n_rows > 0 && step_front_eligible(k_ctx, v_ctx, wk, wv)) {
    // the two writes and the q preparation are independent: one launch does all three
    e = launch_step_front(k_ctx, v_ctx, wk, wv, make_qprep_params(k_ctx, q, q_dtype, s, scale, w), cs);
    if (e != cudaSuccess) return cuda_fail(e, "decode step front launch");
  } else if (n_rows > 0 && step_front_pv_eligible(k_ctx, v_ctx, wk, wv)) {
    e = launch_step_front_pv(k_ctx, v_ctx, wk, wv, make_qprep_params(k_ctx, q, q_dtype, s, scale, w), cs);
    if (e != cudaSuccess) return cuda_fail(e, "decode step front launch");
  } else {
    if (n_rows > 0) {
      if ((e = launch_write(k_ctx, wk, cs)) != cudaSuccess) return cuda_fail(e, "write kernel launch");
      if ((e = launch_write(v_ctx, wv, cs)) != cudaSuccess) return cuda_fail(e, "write kernel launch");
    }
    if ((e = launch_prepare_q(k_ctx, q, q_dtype, s, scale, w, cs)) != cudaSuccess)
      return cuda_fail(e, "prepare_q launch");
  }
  bool fused = false;
  e = launch_partial(k_ctx, v_ctx, (const uint8_t *)k_cache, (const uint8_t *)v_cache, seq_lens, s, nullptr, w,
                     cs, false, out, &fused);
  if (e != cudaSuccess) return cuda_fail(e, "partial launch");
  if (fused) return TQ_OK;
  e = launch_combine(k_ctx, v_ctx, s, out, w, cs);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return TQ_OK;
}

namespace {
size_t dtype_bytes(int dtype) { return dtype == TQ_DTYPE_F32 ? 4 : 2; }
bool dtype_known(int dtype) { return dtype == TQ_DTYPE_F32 || dtype == TQ_DTYPE_BF16 || dtype == TQ_DTYPE_F16; }
// Staging layout of tq_decode_step_host: new K rows, new V rows and q back to back (the
// host order for the one-copy case), then the output at the next 256-byte boundary.
struct HostStaging {
  size_t k_bytes, q_bytes, out_off, out_bytes, total;
};
HostStaging host_staging(int d, int src_dtype, int64_t n_rows, int q_dtype, int B, int Hq) {
  HostStaging h{};
  h.k_bytes = (size_t)n_rows * d * dtype_bytes(src_dtype);
  h.q_bytes = (size_t)B * Hq * d * dtype_bytes(q_dtype);
  h.out_off = (2 * h.k_bytes + h.q_bytes + 255) & ~(size_t)255;
  h.out_bytes = (size_t)B * Hq * d * sizeof(float);
  h.total = h.out_off + h.out_bytes;
  return h;
}
}  // namespace

namespace {
// cuPointerGetAttribute through the runtime's driver entry point (no link to libcuda).
PFN_cuPointerGetAttribute_v4000 pointer_attr_fn() {
  static PFN_cuPointerGetAttribute_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuPointerGetAttribute_v4000>(p);
  });
  return fn;
}

// The device address of the host range [p, p + bytes) when kernels on the current device
// may read and write all of it in place: both ends page-locked host memory of one and the
// same CUDA allocation (so no unmapped gap lies between them), mapped for this device
// contiguously.  Null otherwise (pageable memory, two allocations, no mapping).
void *mapped_host_range(const void *p, size_t bytes) {
  if (!p || bytes == 0) return nullptr;
  const char *b = static_cast<const char *>(p), *e = b + (bytes - 1);
  cudaPointerAttributes a0{}, a1{};
  if (cudaPointerGetAttributes(&a0, b) != cudaSuccess || cudaPointerGetAttributes(&a1, e) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (a0.type != cudaMemoryTypeHost || a1.type != cudaMemoryTypeHost || !a0.devicePointer || !a1.devicePointer)
    return nullptr;
  if (static_cast<const char *>(a1.devicePointer) - static_cast<const char *>(a0.devicePointer) !=
      static_cast<ptrdiff_t>(bytes - 1))
    return nullptr;
  const PFN_cuPointerGetAttribute_v4000 fn = pointer_attr_fn();
  unsigned long long id0 = 0, id1 = 0;
  if (!fn || fn(&id0, CU_POINTER_ATTRIBUTE_BUFFER_ID, (CUdeviceptr)(uintptr_t)b) != CUDA_SUCCESS ||
      fn(&id1, CU_POINTER_ATTRIBUTE_BUFFER_ID, (CUdeviceptr)(uintptr_t)e) != CUDA_SUCCESS || id0 == 0 || id0 != id1)
    return nullptr;
  return a0.devicePointer;
}
}  // namespace

tq_status tq_decode_step_host_staging_size(const tq_ctx *k_ctx, int src_dtype, int64_t n_rows, int q_dtype,
                                           int B, int Hq, size_t *bytes) {
  if (!k_ctx || !bytes) return fail(TQ_ERR_INVALID_ARG, "null context or output");
  if (n_rows < 0 || B < 1 || Hq < 1) return fail(TQ_ERR_INVALID_ARG, "n_rows >= 0, B >= 1 and Hq >= 1 are required");
  if (!dtype_known(q_dtype) || (src_dtype != TQ_DTYPE_F32 && src_dtype != TQ_DTYPE_BF16))
    return fail(TQ_ERR_INVALID_ARG, "unknown dtype");
  *bytes = host_staging(k_ctx->d, src_dtype, n_rows, q_dtype, B, Hq).total;
  return TQ_OK;
}

tq_status tq_decode_step_host(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *inputs_host, int src_dtype,
                              int64_t n_rows, const int64_t *row_ids, int q_dtype, void *k_cache, void *v_cache,
                              const int32_t *seq_lens, int B, int Hq, int Hkv, int L, float scale, float *out_host,
                              void *staging, size_t staging_bytes, void *workspace, size_t workspace_bytes,
                              tq_stream_t stream) {
  if (!k_ctx || !v_ctx) return fail(TQ_ERR_INVALID_ARG, "null context");
  tq_status st = check_current_device(k_ctx->device, "decode");
  if (st != TQ_OK) return st;
  size_t need = 0;
  if ((st = tq_decode_step_host_staging_size(k_ctx, src_dtype, n_rows, q_dtype, B, Hq, &need)) != TQ_OK) return st;
  if (!inputs_host || !out_host) return fail(TQ_ERR_INVALID_ARG, "null host buffer");
  if (!staging || staging_bytes < need) return fail(TQ_ERR_WORKSPACE, "staging smaller than tq_decode_step_host_staging_size()");
  if (!aligned(staging, 256)) return fail(TQ_ERR_ALIGNMENT, "staging must be 256-byte aligned");
  size_t ws_need = 0;  // the shape and workspace checks of the step, before the copy
  if ((st = tq_decode_workspace_size(k_ctx, v_ctx, B, Hq, Hkv, L, &ws_need)) != TQ_OK) return st;
  if (!workspace || workspace_bytes < ws_need) return fail(TQ_ERR_WORKSPACE, "workspace smaller than tq_decode_workspace_size()");
  const HostStaging h = host_staging(k_ctx->d, src_dtype, n_rows, q_dtype, B, Hq);
  // In place when the host buffers are page-locked and mapped (coherent over the
  // chip-to-chip link): the step's kernels read the inputs from and write the output to
  // host memory, so neither copy is issued.  Only where every kernel the step may launch
  // touches those buffers with plain loads and stores: head dimension 128 and at most
  // 256 new rows (the one-launch fronts or the small-batch writes; never the tensor-map
  // write, which takes 2048 rows or more).
  if (k_ctx->d == 128 && n_rows <= 256 && aligned(inputs_host, 16) && aligned(out_host, 4)) {
    const uint8_t *hin = static_cast<const uint8_t *>(mapped_host_range(inputs_host, 2 * h.k_bytes + h.q_bytes));
    float *hout = hin ? static_cast<float *>(mapped_host_range(out_host, h.out_bytes)) : nullptr;
    if (hin && hout)
      return tq_decode_step(k_ctx, v_ctx, hin, hin + h.k_bytes, src_dtype, n_rows, k_ctx->d, row_ids,
                            hin + 2 * h.k_bytes, q_dtype, k_cache, v_cache, seq_lens, B, Hq, Hkv, L, scale, hout,
                            workspace, workspace_bytes, stream);
  }
  uint8_t *dk = static_cast<uint8_t *>(staging), *dv = dk + h.k_bytes, *dq = dv + h.k_bytes;
  float *dout = reinterpret_cast<float *>(dk + h.out_off);
  const cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(dk, inputs_host, 2 * h.k_bytes + h.q_bytes, cudaMemcpyHostToDevice, cs);
  if (e != cudaSuccess) return cuda_fail(e, "input copy");
  st = tq_decode_step(k_ctx, v_ctx, dk, dv, src_dtype, n_rows, k_ctx->d, row_ids, dq, q_dtype, k_cache, v_cache,
                      seq_lens, B, Hq, Hkv, L, scale, dout, workspace, workspace_bytes, stream);
  if (st != TQ_OK) return st;
  e = cudaMemcpyAsync(out_host, dout, h.out_bytes, cudaMemcpyDeviceToHost, cs);
  if (e != cudaSuccess) return cuda_fail(e, "output copy");
  return TQ_OK;
}

tq_status tq_decode_step_num_launches(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int src_dtype, int64_t n_rows,
                                      int B, int Hq, int Hkv, int L, int *n) {
  if (is_d256(k_ctx, v_ctx)) {
    if (!n) return fail(TQ_ERR_INVALID_ARG, "null output");
    D256Shape s;
    tq_status st = check_d256(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
    if (st != TQ_OK) return st;
    if (n_rows < 0) return fail(TQ_ERR_INVALID_ARG, "n_rows < 0");
    *n = 3 + (n_rows > 0 ? 2 : 0);
    return TQ_OK;
  }
  if (!n) return fail(TQ_ERR_INVALID_ARG, "null output");
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (n_rows < 0) return fail(TQ_ERR_INVALID_ARG, "n_rows < 0");
  const int64_t dst_rows = (int64_t)B * Hkv * L;
  const WriteLaunch wk{nullptr, src_dtype, n_rows, D, nullptr, nullptr, dst_rows};
  const int attn = partial_fuses_combine(s) ? 2 : 3;
  const WriteLaunch wv{nullptr, src_dtype, n_rows, D, nullptr, nullptr, dst_rows};
  if (n_rows > 0 && (step_front_eligible(k_ctx, v_ctx, wk, wv) || step_front_pv_eligible(k_ctx, v_ctx, wk, wv)))
    *n = attn;
  else *n = attn + (n_rows > 0 ? 2 : 0);
  return TQ_OK;
}

// ---------------------------------------------------------------- prefill
namespace {
tq_status check_prefill(const tq_ctx *k, const tq_ctx *v, int B, int T, int Hq, int Hkv, int L,
                        PrefillShape *s) {
  if (!k || !v) return fail(TQ_ERR_INVALID_ARG, "null context");
  if (k->device != v->device) return fail(TQ_ERR_INVALID_ARG, "the key and value contexts belong to different devices");
  tq_status st = check_current_device(k->device, "prefill");
  if (st != TQ_OK) return st;
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || L < 1) return fail(TQ_ERR_INVALID_ARG, "B, T, Hq, Hkv and L must be >= 1");
  if (T > L) return fail(TQ_ERR_INVALID_ARG, "the chunk (T queries) must fit in the cache (L rows)");
  if (Hq % Hkv != 0) return fail(TQ_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
  if (k->fmt != TQ_FMT_TURBO4 || v->fmt != TQ_FMT_TURBO4 || k->d != D || v->d != D)
    return fail(TQ_ERR_UNSUPPORTED, "the prefill kernel takes turbo4 keys and values of head dimension 128");
  if (!prefill_shape(k, B, T, Hq, Hkv, L, s))
    return fail(TQ_ERR_UNSUPPORTED, "prefill needs Hq / Hkv dividing 128 and a shape within 32-bit tile counts");
  return TQ_OK;
}
}  // namespace

tq_status tq_prefill_workspace_size(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int T, int Hq,
                                    int Hkv, int L, size_t *bytes) {
  if (!bytes) return fail(TQ_ERR_INVALID_ARG, "null output");
  PrefillShape s;
  tq_status st = check_prefill(k_ctx, v_ctx, B, T, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  *bytes = carve_workspace(s.q, nullptr).bytes;
  return TQ_OK;
}

tq_status tq_prefill_prepare_q(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *q, int q_dtype,
                               int B, int T, int Hq, int Hkv, int L, float scale, void *workspace,
                               size_t workspace_bytes, tq_stream_t stream) {
  PrefillShape s;
  tq_status st = check_prefill(k_ctx, v_ctx, B, T, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (!q) return fail(TQ_ERR_INVALID_ARG, "null q");
  if (q_dtype != TQ_DTYPE_F32 && q_dtype != TQ_DTYPE_BF16 && q_dtype != TQ_DTYPE_F16)
    return fail(TQ_ERR_INVALID_ARG, "bad q dtype");
  if (!aligned(q, 16)) return fail(TQ_ERR_ALIGNMENT, "q must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(TQ_ERR_INVALID_ARG, "scale must be finite");
  if (scale == 0.f) scale = 1.0f / std::sqrt((float)D);
  Workspace w;
  if ((st = check_workspace(s.q, workspace, workspace_bytes, &w)) != TQ_OK) return st;
  cudaError_t e = launch_prepare_q(k_ctx, q, q_dtype, s.q, scale, w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "prepare_q launch");
  return TQ_OK;
}

tq_status tq_prefill_partial(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *k_cache,
                             const void *v_cache, const int32_t *q_start, int B, int T, int Hq,
                             int Hkv, int L, void *workspace, size_t workspace_bytes,
                             tq_stream_t stream) {
  PrefillShape s;
  tq_status st = check_prefill(k_ctx, v_ctx, B, T, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (!k_cache || !v_cache || !q_start) return fail(TQ_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return fail(TQ_ERR_ALIGNMENT, "caches must be 16-byte aligned");
  if (!aligned(q_start, 4)) return fail(TQ_ERR_ALIGNMENT, "q_start must be 4-byte aligned");
  Workspace w;
  if ((st = check_workspace(s.q, workspace, workspace_bytes, &w)) != TQ_OK) return st;
  cudaError_t e = launch_prefill(k_ctx, v_ctx, (const uint8_t *)k_cache, (const uint8_t *)v_cache, q_start, s,
                                 w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return TQ_OK;
}

tq_status tq_prefill_combine(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int T, int Hq, int Hkv,
                             int L, float *out, void *workspace, size_t workspace_bytes,
                             tq_stream_t stream) {
  PrefillShape s;
  tq_status st = check_prefill(k_ctx, v_ctx, B, T, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (!out) return fail(TQ_ERR_INVALID_ARG, "null output");
  if (!aligned(out, 4)) return fail(TQ_ERR_ALIGNMENT, "output must be 4-byte aligned");
  Workspace w;
  if ((st = check_workspace(s.q, workspace, workspace_bytes, &w)) != TQ_OK) return st;
  cudaError_t e = launch_combine_prefill(v_ctx, s, out, w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return TQ_OK;
}

tq_status tq_prefill_attention(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *q, int q_dtype,
                               const void *k_cache, const void *v_cache, const int32_t *q_start,
                               int B, int T, int Hq, int Hkv, int L, float scale, float *out,
                               void *workspace, size_t workspace_bytes, tq_stream_t stream) {
  if (!k_cache || !v_cache || !q_start || !out) return fail(TQ_ERR_INVALID_ARG, "null pointer");
  tq_status st = tq_prefill_prepare_q(k_ctx, v_ctx, q, q_dtype, B, T, Hq, Hkv, L, scale, workspace,
                                      workspace_bytes, stream);
  if (st != TQ_OK) return st;
  st = tq_prefill_partial(k_ctx, v_ctx, k_cache, v_cache, q_start, B, T, Hq, Hkv, L, workspace,
                          workspace_bytes, stream);
  if (st != TQ_OK) return st;
  return tq_prefill_combine(k_ctx, v_ctx, B, T, Hq, Hkv, L, out, workspace, workspace_bytes, stream);
}

tq_status tq_test_ctx_set_device(tq_ctx *ctx, int device) {
  if (!ctx) return fail(TQ_ERR_INVALID_ARG, "null context");
  ctx->device = device;
  return TQ_OK;
}

tq_status tq_test_decode_wait_timeout(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *k_cache,
                                      const void *v_cache, int B, int Hq, int Hkv, int L, void *workspace,
                                      size_t workspace_bytes, tq_stream_t stream) {
  DecodeShape s;
  tq_status st = check_decode_common(k_ctx, v_ctx, B, Hq, Hkv, L, &s);
  if (st != TQ_OK) return st;
  if (s.pv) return fail(TQ_ERR_UNSUPPORTED, "the timeout test runs the turbo4 decode kernel");
  if (!k_cache || !v_cache) return fail(TQ_ERR_INVALID_ARG, "null cache");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return fail(TQ_ERR_ALIGNMENT, "caches must be 16-byte aligned");
  Workspace w;
  if ((st = check_workspace(s, workspace, workspace_bytes, &w)) != TQ_OK) return st;
  cudaError_t e = launch_partial(k_ctx, v_ctx, (const uint8_t *)k_cache, (const uint8_t *)v_cache, nullptr, s,
                                 nullptr, w, (cudaStream_t)stream, true);
  if (e != cudaSuccess) return cuda_fail(e, "partial launch");
  return TQ_OK;
}

}  // extern "C"
