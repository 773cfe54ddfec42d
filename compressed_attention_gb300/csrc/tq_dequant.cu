// Dequantize packed rows to fp32 ("turboquant_plus: how the turbo4 KV format came
// back", section 4: per-element direct extraction, no whole-block cache;
// "TurboQuant fused Triton kernels deep dive", hybrid path that materialises
// history).  One warp per row; lane l produces elements l + 32 m.
//   turbo4 / turbo3: rotated-basis value n * c[idx], optionally mapped back by R^T.
//   prod3: n * (R^T c[idx] + sqrt(pi/2)/d * gamma * S^T sigma)
//          (section 2 bug 2: the QJL term is a product with S^T, not raw signs).
//   vgroup2: code * scale + zero.
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int WARPS = 8;

struct DequantParams {
  const uint8_t *cache;
  int64_t n_rows;
  int fmt;
  int unrotate;
  float c[16];
  const float *r;  // R row-major
  const float *S;  // S row-major
  float qjl_factor;  // 1, or 2/pi for the shrunk QJL estimator
  float *dst;
};

__device__ __forceinline__ int row_bytes_of(int fmt) {
  return fmt == TQ_FMT_TURBO4 ? 68 : (fmt == TQ_FMT_VGROUP2 ? 48 : 56);
}

__device__ __forceinline__ uint32_t idx_of(const uint8_t *row, int fmt, int j) {
  if (fmt == TQ_FMT_TURBO4) return (row[4 + j / 2] >> ((j % 2) * 4)) & 0xFu;
  if (fmt == TQ_FMT_TURBO3) {
    const uint8_t *blk = row + 14 * (j / 32);
    const int jl = j % 32;
    uint32_t v = (blk[2 + jl / 4] >> ((jl % 4) * 2)) & 0x3u;
    if (blk[10 + jl / 8] & (1u << (jl % 8))) v |= 4u;
    return v;
  }
  return (row[(fmt == TQ_FMT_PROD3 ? 8 : 0) + j / 4] >> ((j % 4) * 2)) & 0x3u;
}

__device__ __forceinline__ float norm_of(const uint8_t *row, int fmt, int j) {
  if (fmt == TQ_FMT_TURBO3) {
    const uint8_t *blk = row + 14 * (j / 32);
    const unsigned short bits = (unsigned short)(blk[0] | (blk[1] << 8));
    return __half2float(*reinterpret_cast<const __half *>(&bits));
  }
  return *reinterpret_cast<const float *>(row);
}

__global__ void __launch_bounds__(WARPS * 32) k_dequant(const DequantParams p) {
  __shared__ float yv[WARPS][D];
  __shared__ float sg[WARPS][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t row = (int64_t)blockIdx.x * WARPS + warp; row < p.n_rows;
       row += (int64_t)gridDim.x * WARPS) {
    const uint8_t *rp = p.cache + row * row_bytes_of(p.fmt);
    float out[4];
    if (p.fmt == TQ_FMT_VGROUP2) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int j = lane + 32 * m;
        const __half s = *reinterpret_cast<const __half *>(rp + 32 + 4 * (j / 32));
        const __half z = *reinterpret_cast<const __half *>(rp + 34 + 4 * (j / 32));
        out[m] = (float)idx_of(rp, p.fmt, j) * __half2float(s) + __half2float(z);
      }
    } else {
      const bool prod = p.fmt == TQ_FMT_PROD3;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int j = lane + 32 * m;
        const float c = p.c[idx_of(rp, p.fmt, j)];
        yv[warp][j] = prod ? c : c * norm_of(rp, p.fmt, j);
        if (prod) sg[warp][j] = ((rp[40 + j / 8] >> (j % 8)) & 1u) ? 1.f : -1.f;
      }
      __syncwarp();
      if (!prod && !p.unrotate) {
#pragma unroll
        for (int m = 0; m < 4; ++m) out[m] = yv[warp][lane + 32 * m];
      } else {
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, q[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < D; ++k) {
          const float yk = yv[warp][k];
#pragma unroll
          for (int m = 0; m < 4; ++m) acc[m] = fmaf(p.r[k * D + lane + 32 * m], yk, acc[m]);
          if (prod) {
            const float sk = sg[warp][k];
#pragma unroll
            for (int m = 0; m < 4; ++m) q[m] = fmaf(p.S[k * D + lane + 32 * m], sk, q[m]);
          }
        }
        if (prod) {
          const float n = *reinterpret_cast<const float *>(rp);
          const float gamma = *reinterpret_cast<const float *>(rp + 4);
          const float kq = p.qjl_factor * (1.2533141373155003f / (float)D) * gamma;  // sqrt(pi/2)/d * gamma
#pragma unroll
          for (int m = 0; m < 4; ++m) out[m] = n * (acc[m] + kq * q[m]);
        } else {
#pragma unroll
          for (int m = 0; m < 4; ++m) out[m] = acc[m];
        }
      }
      __syncwarp();
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) p.dst[row * D + lane + 32 * m] = out[m];
  }
}

}  // namespace

cudaError_t launch_dequantize(const tq_ctx *ctx, const uint8_t *cache, int64_t n_rows,
                              int unrotate, float *dst, cudaStream_t st) {
  DequantParams p{};
  p.cache = cache;
  p.n_rows = n_rows;
  p.fmt = ctx->fmt;
  p.unrotate = unrotate;
  for (int k = 0; k < ctx->cb.K; ++k) p.c[k] = ctx->cb.c[k];
  p.r = ctx->d_pi;
  p.S = ctx->d_S;
  p.qjl_factor = ctx->qjl_factor;
  p.dst = dst;
  int64_t want = (n_rows + WARPS - 1) / WARPS;
  int64_t cap = (int64_t)ctx->num_sms * 8;
  const int grid = (int)(want < cap ? want : cap);
  k_dequant<<<grid, WARPS * 32, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tq
