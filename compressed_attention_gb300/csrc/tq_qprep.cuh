// q preparation of the decode (shared by its own kernel and the decode-step front kernel):
// q_rot = R q and, with SKETCH, the QJL sketch S q, each pre-scaled and split into the fp16
// hi + lo tensor-core operands: qhl[q][0..127] = q_rot (hi, lo), qhl[q][128..255] =
// sketch (hi, lo).  A CTA of QWARPS warps takes QWARPS queries, one per warp.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr int QWARPS = 8;  // queries per CTA, one warp each
// dynamic shared memory: R^T (or S^T), the warps' q rows, their fp16 hi + lo rows
constexpr size_t QPREP_SMEM = (size_t)D * D * 4 + QWARPS * D * 4 + QWARPS * 2 * D * 2;

// Stage a 128 x 128 fp32 matrix in shared memory with 16-byte loads, all in flight.
static __device__ __forceinline__ void stage_matrix(float *dst, const float *src) {
  const float4 *s4 = reinterpret_cast<const float4 *>(src);
  float4 *d4 = reinterpret_cast<float4 *>(dst);
  constexpr int N4 = D * D / 4;
  constexpr int PER = N4 / (QWARPS * 32);
  float4 v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) v[i] = s4[threadIdx.x + i * QWARPS * 32];
#pragma unroll
  for (int i = 0; i < PER; ++i) d4[threadIdx.x + i * QWARPS * 32] = v[i];
}

// y = M x for the staged M^T (lane l computes y[l + 32 m]), times mul, scaled by a power
// of two 2^-e so that the largest element lies in [2^13, 2^14), split into fp16 hi and
// lo written to hw[0..127] and hw[128..255].  Returns e.
static __device__ __forceinline__ int transform_split(const float *mt, const float *x, float mul,
                                               __half *hw, int lane) {
  float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
  for (int k = 0; k < D; ++k) {
    const float xk = x[k];
    const float *row = mt + k * D + lane;
#pragma unroll
    for (int m = 0; m < 4; ++m) y[m] = fmaf(row[32 * m], xk, y[m]);
  }
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

// After stage_matrix(qsm, p.rt) and the wait on the previous kernel: CTA cta of n_ctas
// (QWARPS * 32 threads) prepares queries cta * QWARPS .. + QWARPS - 1 and zeroes its share
// of the fused combine's unit counters.
template <bool SKETCH>
static __device__ __forceinline__ void prepare_q_body(const QprepParams &p, int cta, int n_ctas, float *qsm) {
  float *mt = qsm;                       // [128][128]
  float *qv = qsm + D * D;               // [QWARPS][128]
  __half *hs = reinterpret_cast<__half *>(qv + QWARPS * D);  // [QWARPS][2][128]
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
  if (live) {
    const int e = transform_split(mt, qv + warp * D, p.mul, hw, lane);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = src[lane + 32 * i];
    if (lane == 0) {
      p.qsc[2 * qi] = ldexpf(1.0f, e);
      if (!SKETCH) p.qsc[2 * qi + 1] = 0.f;
    }
  }
  if (SKETCH) {
    __syncthreads();  // every warp is done with R^T
    stage_matrix(mt, p.st);
    __syncthreads();
    if (live) {
      __syncwarp();
      const int e = transform_split(mt, qv + warp * D, p.mul_sk, hw, lane);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[128 + lane + 32 * i] = src[lane + 32 * i];
      if (lane == 0) p.qsc[2 * qi + 1] = ldexpf(1.0f, e);
    }
  }
}

}  // namespace tq
