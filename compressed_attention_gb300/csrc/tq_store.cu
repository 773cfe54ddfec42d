// Ring-buffer capture and block-append store ("TurboQuant fused Triton kernels deep dive",
// "write path and codebook": a ring buffer keeps the most recent exact tokens and, when
// it is full, the oldest batch is compressed into the cache, so the decode hot path does
// no per-token quantization; the store appends by blocks).
//
// Device layout of one store (all sequences hold the same number of tokens):
//   k_cache / v_cache  packed rows [B][Hkv][L] (the compressed prefix, tokens [0, flushed))
//   ring_k / ring_v    exact bf16 rows [R][B][Hkv][128], token t in slot t % R (tokens
//                      [flushed, len)); slot-major, so one aligned block of F = R / 2
//                      slots is one contiguous source for one SET_ROWS launch
// Appending copies the new tokens into their slots; when the ring is full the oldest
// block (F tokens of every (sequence, KV head)) is quantized by one SET_ROWS launch into
// cache rows [flushed, flushed + F) and flushed advances by F.  Decode attends over both
// parts: the split-K decode over the compressed prefix and one exact partial over the
// ring tail (k_tail_partial, here), merged by the same combine.
#include <cuda_runtime.h>
#include <math.h>

#include <new>

#include "tq.h"
#include "tq_decode_common.cuh"
#include "tq_device.cuh"
#include "tq_internal.h"

struct tq_store {
  const tq_ctx *k = nullptr, *v = nullptr;
  int B = 0, Hkv = 0, L = 0, R = 0, F = 0;
  int device = 0;
  uint8_t *k_cache = nullptr, *v_cache = nullptr;
  uint16_t *ring_k = nullptr, *ring_v = nullptr;
  int64_t *row_ids = nullptr;  // destinations of one flush block, [F * B * Hkv]
  int32_t *lens = nullptr;     // per-sequence length of the compressed prefix, [B]
  int64_t len = 0;             // tokens appended per sequence
  int64_t flushed = 0;         // of which compressed
};

namespace tq {
namespace {

constexpr int TAIL_WARPS = 8;

// Copy tokens [t0, t0 + m) of src [B][Hkv][n][128] bf16 into ring slots (pos0 + i) % R.
__global__ void k_ring_put(uint16_t *ring, const uint16_t *src, int BH, int n, int t0, int m,
                           int64_t pos0, int R) {
  const int64_t total = (int64_t)m * BH * 16;  // 16-byte chunks
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i & 15);
    const int64_t row = i >> 4;
    const int u = (int)(row % BH), tk = (int)(row / BH);
    const uint4 v = reinterpret_cast<const uint4 *>(src + ((int64_t)u * n + t0 + tk) * D)[c];
    const int64_t slot = (pos0 + tk) % R;
    reinterpret_cast<uint4 *>(ring + (slot * BH + u) * D)[c] = v;
  }
}

// Destinations of the flush block starting at token `first`: ring row i * BH + u (block
// slot i, unit u) goes to cache row u * L + first + i; and the compressed length of every
// sequence becomes first + F.
__global__ void k_flush_ids(int64_t *ids, int32_t *lens, int F, int BH, int B, int L, int64_t first) {
  const int total = F * BH;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int u = i % BH, s = i / BH;
    ids[i] = (int64_t)u * L + first + s;
  }
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x)
    lens[b] = (int32_t)(first + F);
}

struct TailParams {
  const void *q;
  int q_dtype;
  const uint16_t *ring_k, *ring_v;
  int B, Hq, Hkv, R;
  int64_t first;    // position of the oldest exact token
  int n_tail;       // exact tokens per sequence
  float mul;        // log2(e) * scale
  const float *r;   // value rotation R (row-major), or null for unrotated values
  float vscale;     // 2^P_SHIFT * alpha_V (1 for unrotated values)
  float *part;
  int n_part, slot;
};

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// One warp per (batch, q-head): the partial (max, sum, acc) of the exact ring tokens, in the
// decode's conventions: scores in log2 units, acc = sum 2^(s - M) (R v) 2^P_SHIFT alpha_V,
// so the combine merges it with the split-K partials and un-rotates once.
__global__ void __launch_bounds__(TAIL_WARPS * 32) k_tail_partial(const TailParams p) {
  __shared__ float accs[TAIL_WARPS][D];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x * TAIL_WARPS + warp;
  const bool live = bh < p.B * p.Hq;
  const int b = bh / p.Hq, h = bh % p.Hq, kv = (h * p.Hkv) / p.Hq;
  const int BH = p.B * p.Hkv, u = b * p.Hkv + kv;
  float qv[4] = {0.f, 0.f, 0.f, 0.f};
  if (live) {
    if (p.q_dtype == TQ_DTYPE_F32) {
      const float4 v = reinterpret_cast<const float4 *>(p.q)[(size_t)bh * 32 + lane];
      qv[0] = v.x, qv[1] = v.y, qv[2] = v.z, qv[3] = v.w;
    } else {
      const uint2 v = reinterpret_cast<const uint2 *>(p.q)[(size_t)bh * 32 + lane];
      const uint32_t w[4] = {v.x & 0xFFFFu, v.x >> 16, v.y & 0xFFFFu, v.y >> 16};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (p.q_dtype == TQ_DTYPE_BF16) {
          qv[e] = bf16f(w[e]);
        } else {
          const unsigned short us = (unsigned short)w[e];
          qv[e] = __half2float(*reinterpret_cast<const __half *>(&us));
        }
      }
    }
  }
  // scores: lane l holds dims 4l..4l+3 of q and of each key
  auto score = [&](int t) {
    const int64_t slot = (p.first + t) % p.R;
    const uint2 kw = reinterpret_cast<const uint2 *>(p.ring_k + (slot * BH + u) * D)[lane];
    float s = qv[0] * bf16f(kw.x & 0xFFFFu);
    s = fmaf(qv[1], bf16f(kw.x >> 16), s);
    s = fmaf(qv[2], bf16f(kw.y & 0xFFFFu), s);
    s = fmaf(qv[3], bf16f(kw.y >> 16), s);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(FULL_MASK, s, o);
    return s * p.mul;
  };
  float M = -INFINITY;
  if (live)
    for (int t = 0; t < p.n_tail; ++t) M = fmaxf(M, score(t));
  float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (live) {
    for (int t = 0; t < p.n_tail; ++t) {
      const float w = exp2f(score(t) - M);
      l += w;
      const int64_t slot = (p.first + t) % p.R;
      const uint2 vw = reinterpret_cast<const uint2 *>(p.ring_v + (slot * BH + u) * D)[lane];
      acc[0] = fmaf(w, bf16f(vw.x & 0xFFFFu), acc[0]);
      acc[1] = fmaf(w, bf16f(vw.x >> 16), acc[1]);
      acc[2] = fmaf(w, bf16f(vw.y & 0xFFFFu), acc[2]);
      acc[3] = fmaf(w, bf16f(vw.y >> 16), acc[3]);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) accs[warp][4 * lane + e] = acc[e];
  __syncwarp();
  if (!live) return;
  float *dst = p.part + ((size_t)bh * p.n_part + p.slot) * PARTIAL_FLOATS;
  const bool any = p.n_tail > 0;
#pragma unroll
  for (int m = 0; m < 4; ++m) {  // output j = lane + 32 m of R acc (or acc itself)
    const int j = lane + 32 * m;
    float o = 0.f;
    if (p.r) {
      const float *row = p.r + (size_t)j * D;
      for (int k = 0; k < D; ++k) o = fmaf(row[k], accs[warp][k], o);
    } else {
      o = accs[warp][j];
    }
    dst[6 + j] = any ? o * p.vscale : 0.f;
  }
  if (lane == 0) {
    dst[0] = any ? M : -INFINITY;
    dst[1] = any ? l : 0.f;
    dst[2] = dst[3] = dst[4] = dst[5] = 0.f;
  }
}

tq_status fail(tq_status s, const char *msg) {
  set_error("%s", msg);
  return s;
}
tq_status cuda_fail(cudaError_t e, const char *what) {
  set_error("%s: %s", what, cudaGetErrorString(e));
  return TQ_ERR_CUDA;
}

// The decode geometry of a store: split-K over the compressed capacity (per-sequence
// lengths = the compressed prefix), plus one more partial slot per head for the ring.
tq_status store_shape(const tq_store *st, int Hq, DecodeShape *s) {
  if (Hq < 1 || Hq % st->Hkv != 0) return fail(TQ_ERR_INVALID_ARG, "Hq must be a positive multiple of Hkv");
  if (!decode_shape(st->k, st->v, st->B, Hq, st->Hkv, st->L, s)) return fail(TQ_ERR_UNSUPPORTED, "shape too large");
  s->n_part += 1;
  s->tail_slot = s->n_part - 1;
  s->no_main = st->flushed == 0;
  return TQ_OK;
}

tq_status flush_block(tq_store *st, cudaStream_t cs) {
  if (st->flushed + st->F > st->L) return fail(TQ_ERR_INVALID_ARG, "store full: the compressed cache holds L tokens per sequence");
  const int BH = st->B * st->Hkv;
  const int64_t slot0 = st->flushed % st->R;
  k_flush_ids<<<(max(st->F * BH, st->B) + 255) / 256, 256, 0, cs>>>(st->row_ids, st->lens, st->F, BH, st->B, st->L, st->flushed);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "flush ids launch");
  const int64_t rows = (int64_t)st->F * BH, cache_rows = (int64_t)BH * st->L;
  for (int t = 0; t < 2; ++t) {
    WriteLaunch w{(t ? st->ring_v : st->ring_k) + slot0 * BH * D, TQ_DTYPE_BF16, rows, D, st->row_ids,
                  t ? st->v_cache : st->k_cache, cache_rows};
    if ((e = launch_write(t ? st->v : st->k, w, cs)) != cudaSuccess) return cuda_fail(e, "flush write launch");
  }
  st->flushed += st->F;
  return TQ_OK;
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" {

tq_status tq_store_create(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int Hkv, int L, int ring_tokens,
                          tq_store **out) {
  if (!out) return fail(TQ_ERR_INVALID_ARG, "null output");
  *out = nullptr;
  if (!k_ctx || !v_ctx) return fail(TQ_ERR_INVALID_ARG, "null context");
  if (B < 1 || Hkv < 1 || L < 1) return fail(TQ_ERR_INVALID_ARG, "B, Hkv and L must be >= 1");
  if (ring_tokens < 2 || ring_tokens % 2 != 0 || ring_tokens > 4096)
    return fail(TQ_ERR_INVALID_ARG, "ring_tokens must be even, in [2, 4096]");
  if (B > 1024) return fail(TQ_ERR_UNSUPPORTED, "at most 1024 sequences");
  DecodeShape probe;
  if (!decode_pair_supported(k_ctx, v_ctx) || !decode_shape(k_ctx, v_ctx, B, Hkv, Hkv, L, &probe))
    return fail(TQ_ERR_UNSUPPORTED, "no decode kernel for this (key, value) format pair or shape");
  if (k_ctx->device != v_ctx->device) return fail(TQ_ERR_INVALID_ARG, "contexts on different devices");
  if (tq_status cs = check_current_device(k_ctx->device, "tq_store_create")) return cs;
  tq_store *st = new (std::nothrow) tq_store();
  if (!st) return fail(TQ_ERR_CUDA, "host allocation failed");
  st->k = k_ctx, st->v = v_ctx, st->B = B, st->Hkv = Hkv, st->L = L, st->R = ring_tokens, st->F = ring_tokens / 2;
  st->device = k_ctx->device;
  const int64_t BH = (int64_t)B * Hkv;
  cudaError_t e = cudaSuccess;
  auto alloc = [&](void **p, size_t bytes) {
    if (e == cudaSuccess) e = cudaMalloc(p, bytes);
    if (e == cudaSuccess) e = cudaMemset(*p, 0, bytes);
  };
  alloc((void **)&st->k_cache, tq_cache_bytes(k_ctx->fmt, BH * L));
  alloc((void **)&st->v_cache, tq_cache_bytes(v_ctx->fmt, BH * L));
  alloc((void **)&st->ring_k, (size_t)ring_tokens * BH * D * 2);
  alloc((void **)&st->ring_v, (size_t)ring_tokens * BH * D * 2);
  alloc((void **)&st->row_ids, (size_t)st->F * BH * sizeof(int64_t));
  alloc((void **)&st->lens, (size_t)B * sizeof(int32_t));
  if (e != cudaSuccess) {
    tq_store_destroy(st);
    return cuda_fail(e, "store allocation");
  }
  *out = st;
  return TQ_OK;
}

tq_status tq_store_destroy(tq_store *st) {
  if (!st) return TQ_OK;
  cudaFree(st->k_cache);
  cudaFree(st->v_cache);
  cudaFree(st->ring_k);
  cudaFree(st->ring_v);
  cudaFree(st->row_ids);
  cudaFree(st->lens);
  delete st;
  return TQ_OK;
}

tq_status tq_store_append(tq_store *st, const void *k_new, const void *v_new, int n, tq_stream_t stream) {
  if (!st) return fail(TQ_ERR_INVALID_ARG, "null store");
  if (n < 0) return fail(TQ_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return TQ_OK;
  if (tq_status cs = check_current_device(st->device, "tq_store_append")) return cs;
  if (!k_new || !v_new) return fail(TQ_ERR_INVALID_ARG, "null source");
  if (((uintptr_t)k_new | (uintptr_t)v_new) % 16) return fail(TQ_ERR_ALIGNMENT, "sources must be 16-byte aligned");
  // every flush this append needs must fit: tokens beyond the last flush stay in the ring
  const int64_t end = st->len + n, flush_to = end > st->R ? ((end - st->R + st->F - 1) / st->F) * st->F : 0;
  if (flush_to > st->L) return fail(TQ_ERR_INVALID_ARG, "store full: the compressed cache holds L tokens per sequence");
  const cudaStream_t cs = (cudaStream_t)stream;
  const int BH = st->B * st->Hkv;
  int t0 = 0;
  while (t0 < n) {
    if (st->len - st->flushed == st->R) {  // the ring is full: compress its oldest block
      tq_status s = flush_block(st, cs);
      if (s != TQ_OK) return s;
    }
    const int room = (int)(st->R - (st->len - st->flushed));
    const int m = n - t0 < room ? n - t0 : room;
    const int64_t chunks = (int64_t)m * BH * 16;
    const int grid = (int)((chunks + 255) / 256 < 4096 ? (chunks + 255) / 256 : 4096);
    for (int t = 0; t < 2; ++t)
      k_ring_put<<<grid, 256, 0, cs>>>(t ? st->ring_v : st->ring_k, (const uint16_t *)(t ? v_new : k_new), BH, n,
                                      t0, m, st->len, st->R);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "ring copy launch");
    st->len += m;
    t0 += m;
  }
  return TQ_OK;
}

tq_status tq_store_state(const tq_store *st, int64_t *len, int64_t *flushed, const void **k_cache,
                         const void **v_cache) {
  if (!st) return fail(TQ_ERR_INVALID_ARG, "null store");
  if (len) *len = st->len;
  if (flushed) *flushed = st->flushed;
  if (k_cache) *k_cache = st->k_cache;
  if (v_cache) *v_cache = st->v_cache;
  return TQ_OK;
}

tq_status tq_store_workspace_size(const tq_store *st, int Hq, size_t *bytes) {
  if (!st || !bytes) return fail(TQ_ERR_INVALID_ARG, "null argument");
  DecodeShape s;
  tq_status r = store_shape(st, Hq, &s);
  if (r != TQ_OK) return r;
  *bytes = carve_workspace(s, nullptr).bytes;
  return TQ_OK;
}

tq_status tq_store_decode(const tq_store *st, const void *q, int q_dtype, int Hq, float scale, float *out,
                          void *workspace, size_t workspace_bytes, tq_stream_t stream) {
  if (!st) return fail(TQ_ERR_INVALID_ARG, "null store");
  if (tq_status cs = check_current_device(st->device, "tq_store_decode")) return cs;
  if (!q || !out || !workspace) return fail(TQ_ERR_INVALID_ARG, "null pointer");
  if (st->len == 0) return fail(TQ_ERR_INVALID_ARG, "the store is empty");
  if (q_dtype != TQ_DTYPE_F32 && q_dtype != TQ_DTYPE_BF16 && q_dtype != TQ_DTYPE_F16)
    return fail(TQ_ERR_INVALID_ARG, "bad q dtype");
  if ((uintptr_t)q % 16 || (uintptr_t)out % 4) return fail(TQ_ERR_ALIGNMENT, "q must be 16-byte, out 4-byte aligned");
  if ((uintptr_t)workspace % 256) return fail(TQ_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (!std::isfinite(scale)) return fail(TQ_ERR_INVALID_ARG, "scale must be finite");
  if (scale == 0.f) scale = 1.0f / std::sqrt((float)D);
  DecodeShape s;
  tq_status r = store_shape(st, Hq, &s);
  if (r != TQ_OK) return r;
  Workspace w = carve_workspace(s, workspace);
  if (workspace_bytes < w.bytes) return fail(TQ_ERR_WORKSPACE, "workspace smaller than tq_store_workspace_size()");
  const cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  if (!s.no_main) {  // the compressed prefix: q preparation and split-K partials
    if ((e = launch_prepare_q(st->k, q, q_dtype, s, scale, w, cs)) != cudaSuccess) return cuda_fail(e, "prepare_q launch");
    if ((e = launch_partial(st->k, st->v, st->k_cache, st->v_cache, st->lens, s, nullptr, w, cs)) != cudaSuccess)
      return cuda_fail(e, "partial launch");
  }
  TailParams tp{};
  tp.q = q, tp.q_dtype = q_dtype;
  tp.ring_k = st->ring_k, tp.ring_v = st->ring_v;
  tp.B = st->B, tp.Hq = Hq, tp.Hkv = st->Hkv, tp.R = st->R;
  tp.first = st->flushed;
  tp.n_tail = (int)(st->len - st->flushed);
  tp.mul = LOG2E * scale;
  const bool vgroup = st->v->fmt == TQ_FMT_VGROUP2;
  tp.r = vgroup ? nullptr : st->v->d_pi;
  tp.vscale = exp2f(P_SHIFT) * (vgroup ? 1.0f : st->v->f16.alpha);
  tp.part = w.partials, tp.n_part = s.n_part, tp.slot = s.tail_slot;
  const int heads = st->B * Hq;
  if ((e = launch_pdl(k_tail_partial, dim3((heads + TAIL_WARPS - 1) / TAIL_WARPS), dim3(TAIL_WARPS * 32), 0, cs, tp)) !=
      cudaSuccess)
    return cuda_fail(e, "tail launch");
  if ((e = launch_combine(st->k, st->v, s, out, w, cs)) != cudaSuccess) return cuda_fail(e, "combine launch");
  return TQ_OK;
}

}  // extern "C"
