// tq_decode_attention_static: the fused decode with its scratch in a fixed-size area of
// static device memory, so the call allocates nothing.
//
// Some callers cannot hand the library a workspace or let it allocate one: plugin code
// inside a host framework that owns every byte of device memory (its allocator must
// account for all of it, and a private cudaMalloc next to it fragments or exceeds the
// budget), and step loops that must not stall, where cudaMalloc / cudaFree can wait for
// the whole device.  For them the scratch of the decode (rotated queries and the split-K
// partials) lives in g_decode_scratch below, which the CUDA module carries once per
// device.  The call itself does no allocation of any kind, here or in the kernels.
//
// The arithmetic is exactly that of tq_decode_attention: this file only resolves the
// static area's address and forwards to it.
#include <cuda_runtime.h>

#include <mutex>

#include "tq_internal.h"

using namespace tq;

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[TQ_STATIC_WORKSPACE_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[MAX_DEVICES] = {};

// Device address of g_decode_scratch on `device`, resolved once per device.  The caller
// has checked that `device` is current, so the lookup (which may load the module on it)
// needs no switch of the current device.
tq_status scratch_on(int device, void **ptr) {
  if (device < 0 || device >= MAX_DEVICES) {
    set_error("tq_decode_attention_static: device %d beyond the %d devices it supports", device,
              MAX_DEVICES);
    return TQ_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[device]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) {
      set_error("tq_decode_attention_static: static scratch lookup on device %d: %s", device,
                cudaGetErrorString(e));
      return TQ_ERR_CUDA;
    }
    g_scratch_ptr[device] = p;
  }
  *ptr = g_scratch_ptr[device];
  return TQ_OK;
}

}  // namespace

extern "C" {

tq_status tq_decode_attention_static(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *q,
                                     int q_dtype, const void *k_cache, const void *v_cache,
                                     const int32_t *seq_lens, int B, int Hq, int Hkv, int L,
                                     float scale, float *out, tq_stream_t stream) {
  if (!k_ctx || !v_ctx) {
    set_error("tq_decode_attention_static: null context");
    return TQ_ERR_INVALID_ARG;
  }
  // (the size query also checks that both contexts belong to the current device)
  size_t need = 0;
  tq_status st = tq_decode_workspace_size(k_ctx, v_ctx, B, Hq, Hkv, L, &need);
  if (st != TQ_OK) return st;
  if (need > (size_t)TQ_STATIC_WORKSPACE_BYTES) {
    set_error("tq_decode_attention_static: this shape needs %zu bytes of scratch, the static area "
              "holds %zu; use tq_decode_attention with a caller workspace",
              need, (size_t)TQ_STATIC_WORKSPACE_BYTES);
    return TQ_ERR_WORKSPACE;
  }
  void *ws = nullptr;
  if ((st = scratch_on(k_ctx->device, &ws)) != TQ_OK) return st;
  return tq_decode_attention(k_ctx, v_ctx, q, q_dtype, k_cache, v_cache, seq_lens, B, Hq, Hkv, L,
                             scale, out, nullptr, ws, (size_t)TQ_STATIC_WORKSPACE_BYTES, stream);
}

size_t tq_static_workspace_bytes(void) { return (size_t)TQ_STATIC_WORKSPACE_BYTES; }

}  // extern "C"
