// q preparation of the decode (shared by its own kernel and the decode-step front kernels):
// q_rot = R q and, with SKETCH, the QJL sketch S q, each pre-scaled and split into the fp16
// hi + lo tensor-core operands: qhl[q][0..127] = q_rot (hi, lo), qhl[q][128..255] =
// sketch (hi, lo).  A CTA of QWARPS warps takes QWARPS queries: for the products warp w
// computes outputs 16w .. 16w+15 of every query of the CTA from R (row-major, padded rows
// in shared memory), so each row of R is read from shared memory once per CTA rather than
// once per query; then warp w scales and splits query w.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int QWARPS = 8;  // queries per CTA
constexpr int RPAD = D + 4;  // padded row of a staged matrix: rows 16 apart share no bank
// dynamic shared memory: R (or S) with padded rows, the CTA's q rows, their products, the
// fp16 hi + lo rows
constexpr size_t QPREP_SMEM = (size_t)D * RPAD * 4 + 2 * QWARPS * D * 4 + QWARPS * 2 * D * 2;

// One 16-byte asynchronous copy global -> shared (both 16-byte aligned).
static __device__ __forceinline__ void cp16_async(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// Stage a 128 x 128 fp32 matrix (row-major) in shared memory with rows of `pitch` floats
// (D: packed; RPAD: padded, so that rows 16 apart share no bank), by every thread of the
// CTA with 16-byte asynchronous copies, all in flight at once; each thread waits for its
// own copies, so the caller's next barrier makes the matrix visible to the CTA.
static __device__ __forceinline__ void stage_matrix_pitch(float *dst, const float *src, int pitch) {
  for (int i = threadIdx.x; i < D * D / 4; i += blockDim.x)
    cp16_async(dst + (i / (D / 4)) * pitch + 4 * (i % (D / 4)), src + 4 * i);
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
}
static __device__ __forceinline__ void stage_matrix(float *dst, const float *src) { stage_matrix_pitch(dst, src, D); }
static __device__ __forceinline__ void stage_rows_padded(float *dst, const float *src) {
  stage_matrix_pitch(dst, src, RPAD);
}

// ys[q][j] = (M x_q)_j for the CTA's QWARPS queries xs[q][0..127] and the staged M (padded
// rows): warp w takes outputs j = 16w + (lane & 15) of queries 4 (lane >> 4) .. + 3, each a
// chain of fused multiply-adds over k in order (as one query per warp would give).
static __device__ __forceinline__ void transform_cta(const float *m, const float *xs, float *ys, int warp,
                                                     int lane) {
  const int j = 16 * warp + (lane & 15), q0 = 4 * (lane >> 4);
  const float *mr = m + j * RPAD;
  float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int k = 0; k < D; k += 4) {
    const float4 r = *reinterpret_cast<const float4 *>(mr + k);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 x = *reinterpret_cast<const float4 *>(xs + (q0 + i) * D + k);
      y[i] = fmaf(r.x, x.x, y[i]);
      y[i] = fmaf(r.y, x.y, y[i]);
      y[i] = fmaf(r.z, x.z, y[i]);
      y[i] = fmaf(r.w, x.w, y[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) ys[(q0 + i) * D + j] = y[i];
}

// Query `warp`'s products ys[warp][0..127] times mul, scaled by a power of two 2^-e so that
// the largest element lies in [2^13, 2^14), split into fp16 hi and lo written to
// hw[0..127] and hw[128..255].  Returns e.
static __device__ __forceinline__ int scale_split(const float *yrow, float mul, __half *hw, int lane) {
  float y[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) y[m] = yrow[lane + 32 * m];
  float amax = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    y[m] *= mul;
    amax = fmaxf(amax, fabsf(y[m]));
  }
#pragma unroll
  for (int h = 16; h >= 1; h >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, h));
  int e = 0;
  if (amax > 0.f && isfinite(amax)) e = ilogbf(amax) - 13;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float v = ldexpf(y[m], -e);
    const __half h = __float2half_rn(v);
    hw[lane + 32 * m] = h;
    hw[D + lane + 32 * m] = __float2half_rn(v - __half2float(h));
  }
  return e;
}

// After stage_rows_padded(qsm, p.r) and the wait on the previous kernel: CTA cta of n_ctas
// (QWARPS * 32 threads) prepares queries cta * QWARPS .. + QWARPS - 1 and zeroes its share
// of the fused combine's unit counters.
template <bool SKETCH>
static __device__ __forceinline__ void prepare_q_body(const QprepParams &p, int cta, int n_ctas, float *qsm) {
  float *mt = qsm;                       // [128][RPAD]
  float *qv = qsm + D * RPAD;            // [QWARPS][128]
  float *yv = qv + QWARPS * D;           // [QWARPS][128]
  __half *hs = reinterpret_cast<__half *>(yv + QWARPS * D);  // [QWARPS][2][128]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qi = cta * QWARPS + warp;
  const bool live = qi < p.n_q;
  float x[4] = {0.f, 0.f, 0.f, 0.f};
  if (live) {
    if (p.q_dtype == TQ_DTYPE_F32) {
      const float4 v = reinterpret_cast<const float4 *>(p.q)[(size_t)qi * 32 + lane];
      x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
    } else {
      const uint2 v = reinterpret_cast<const uint2 *>(p.q)[(size_t)qi * 32 + lane];
      const uint32_t w[4] = {v.x & 0xFFFFu, v.x >> 16, v.y & 0xFFFFu, v.y >> 16};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (p.q_dtype == TQ_DTYPE_BF16) {
          x[e] = bf16_bits_to_f32(w[e]);
        } else {
          const unsigned short us = (unsigned short)w[e];
          x[e] = __half2float(*reinterpret_cast<const __half *>(&us));
        }
      }
    }
  }
  *reinterpret_cast<float4 *>(&qv[warp * D + 4 * lane]) = make_float4(x[0], x[1], x[2], x[3]);
  // after the wait: the previous split-K launch may still have been counting
  for (int i = cta * blockDim.x + threadIdx.x; i < p.n_units; i += n_ctas * blockDim.x) p.unit_done[i] = 0;
  __syncthreads();
  __half *hw = hs + warp * 2 * D;
  uint32_t *dst = p.qhl + (size_t)qi * 256;
  const uint32_t *src = reinterpret_cast<const uint32_t *>(hw);
  transform_cta(mt, qv, yv, warp, lane);
  __syncthreads();
  if (live) {
    const int e = scale_split(yv + warp * D, p.mul, hw, lane);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = src[lane + 32 * i];
    if (lane == 0) {
      p.qsc[2 * qi] = ldexpf(1.0f, e);
      if (!SKETCH) p.qsc[2 * qi + 1] = 0.f;
    }
  }
  if (SKETCH) {
    __syncthreads();  // every warp is done with R and with its products
    stage_rows_padded(mt, p.s);
    __syncthreads();
    transform_cta(mt, qv, yv, warp, lane);
    __syncthreads();
    if (live) {
      __syncwarp();
      const int e = scale_split(yv + warp * D, p.mul_sk, hw, lane);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[128 + lane + 32 * i] = src[lane + 32 * i];
      if (lane == 0) p.qsc[2 * qi + 1] = ldexpf(1.0f, e);
    }
  }
}

}  // namespace tq
