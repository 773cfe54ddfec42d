// Fused decode attention over the packed cache ("TurboQuant fused Triton kernels
// deep dive", tricks 1-3): q is rotated once, every key is scored straight from
// its 4-bit indices, online softmax runs over key tiles split across the SMs,
// values are dequantized in registers, and the output is un-rotated once.
//
// Three launches:
//   k_prepare_q  q_rot = R q (one warp per query), pre-scaled by
//                log2(e) * scale / alpha and by a power of two, split into fp16
//                hi + lo parts (the tensor-core A operand).
//   k_partial_*  one CTA per (batch, KV head, head group, key split): a producer
//                warp streams 64-key tiles of the K and V caches into shared
//                memory with 1-D bulk async copies on an mbarrier ring; four
//                consumer warps each take 16 keys of a tile, decode the nibbles
//                to fp16 centroids with byte permutes, and run the score and PV
//                products as m16n8k16 MMAs with fp32 accumulators.
//   k_combine    log-sum-exp merge of the splits, 1/sum, un-rotation R^T o.
//
// Operand layout of the MMAs (one warp, 16 keys, up to 8 q-heads of one KV head):
//   score  S[16 x 8 keys] = Q[16 x 128] * K_hat^T : row h = q_hi of head h, row
//          h+8 = q_lo of head h, so S[h] + S[h+8] is the score at fp32 accuracy.
//   PV     O[16 x 128] += P[16 x 16 keys] * V_hat : row h = p_hi, row h+8 = p_lo.
//   The score accumulator fragment of two key tiles is exactly the A fragment
//   of the PV product, so probabilities never leave registers.
// Centroids enter as fp16 values alpha * |c| with the sign applied from the
// index; alpha (chosen on the host) minimises the fp16 rounding error of the
// table and is divided out through q and in the combine.
#include <math.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int TILE = 64;              // keys per pipeline stage
constexpr int CWARPS = 4;             // consumer warps (16 keys each per tile)
constexpr int NTHREADS = (CWARPS + 1) * 32;
constexpr int NSTAGE = 4;             // pipeline depth
constexpr int T4_ROW = 68;
constexpr int STAGE_BUF = 4416;       // >= 64 * 68 + 2 * 16, multiple of 32
constexpr float P_SHIFT = 14.0f;      // p' = 2^14 * exp2(.) keeps fp16 normal
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// 8 packed 4-bit indices -> 8 fp16 centroid values as four fp16x2 words.
// Magnitude index m = idx for idx < 8 (negative centroids), 15 - idx otherwise;
// sign is negative when bit 3 of the index is clear.  SEL0 / SEL1 choose how the
// looked-up bytes pair up: (0,1),(2,3) for dims of one key, (0,2),(1,3) for the
// same dim of two keys after a byte interleave.
template <uint32_t SEL0, uint32_t SEL1>
__device__ __forceinline__ void decode8(uint32_t x, const uint32_t (&lo)[2],
                                        const uint32_t (&hi)[2], uint32_t (&r)[4]) {
  const uint32_t t = x & 0x88888888u;
  const uint32_t m = (x ^ (t - (t >> 3))) & 0x77777777u;
  const uint32_t x4 = x << 4;
  const uint32_t pos_a = prmt(x, x4, 0x9D8Cu);  // 0xFF per byte where nibble 0..3 >= 8
  const uint32_t pos_b = prmt(x, x4, 0xBFAEu);  // nibbles 4..7
  const uint32_t mh = m >> 16;
  const uint32_t lo_a = prmt(lo[0], lo[1], m);
  const uint32_t lo_b = prmt(lo[0], lo[1], mh);
  const uint32_t hi_a = prmt(hi[0], hi[1], m) | (~pos_a & 0x80808080u);
  const uint32_t hi_b = prmt(hi[0], hi[1], mh) | (~pos_b & 0x80808080u);
  r[0] = prmt(lo_a, hi_a, SEL0);
  r[1] = prmt(lo_a, hi_a, SEL1);
  r[2] = prmt(lo_b, hi_b, SEL0);
  r[3] = prmt(lo_b, hi_b, SEL1);
}

struct QprepParams {
  const void *q;
  int q_dtype;
  int n_q;            // B * Hq
  const float *rt;    // R^T, fp32 [128][128] (row k = column k of R)
  float mul;          // log2(e) * scale / alpha_K
  uint32_t *qhl;
  float *qsc;
};

constexpr int QWARPS = 8;

__global__ void __launch_bounds__(QWARPS * 32) k_prepare_q(const QprepParams p) {
  __shared__ __align__(16) float qv[QWARPS][D];
  __shared__ __align__(16) __half hs[QWARPS][2][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qi = blockIdx.x * QWARPS + warp;
  if (qi >= p.n_q) return;
  float x[4];
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
  *reinterpret_cast<float4 *>(&qv[warp][4 * lane]) = make_float4(x[0], x[1], x[2], x[3]);
  __syncwarp();
  float y[4] = {0.f, 0.f, 0.f, 0.f};  // q_rot[j], j = lane + 32 m
  for (int k = 0; k < D; ++k) {
    const float qk = qv[warp][k];
    const float *row = p.rt + k * D + lane;
#pragma unroll
    for (int m = 0; m < 4; ++m) y[m] = fmaf(row[32 * m], qk, y[m]);
  }
  float amax = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    y[m] *= p.mul;
    amax = fmaxf(amax, fabsf(y[m]));
  }
#pragma unroll
  for (int h = 16; h >= 1; h >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, h));
  int e = 0;
  if (amax > 0.f && isfinite(amax)) e = ilogbf(amax) - 13;  // amax * 2^-e in [2^13, 2^14)
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float v = ldexpf(y[m], -e);
    const __half h = __float2half_rn(v);
    hs[warp][0][lane + 32 * m] = h;
    hs[warp][1][lane + 32 * m] = __float2half_rn(v - __half2float(h));
  }
  __syncwarp();
  uint32_t *dst = p.qhl + (size_t)qi * 256;
  const uint32_t *src = reinterpret_cast<const uint32_t *>(&hs[warp][0][0]);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = src[lane + 32 * i];
  if (lane == 0) {
    p.qsc[2 * qi] = ldexpf(1.0f, e);
    p.qsc[2 * qi + 1] = 0.f;
  }
}

struct PartialParams {
  const uint8_t *kc;
  const uint8_t *vc;
  const int32_t *seq_lens;
  int B, Hq, Hkv, L, gq, n_hg, n_split, chunk;
  const uint32_t *qhl;
  const float *qsc;
  float *part;
  float *scores;
  uint32_t klo[2], khi[2], vlo[2], vhi[2];
  int32_t *status;
};

struct SmemPartial {
  uint8_t kbuf[NSTAGE][STAGE_BUF];
  uint8_t vbuf[NSTAGE][STAGE_BUF];
  uint64_t full[NSTAGE];
  uint64_t empty[NSTAGE];
  float mw[CWARPS][8];
  float lw[CWARPS][8];
  float osm[8][D];
  int abort_flag;
  int first_unconsumed;
  int issued;
};

template <bool SCORES>
__global__ void __launch_bounds__(NTHREADS, 2) k_partial_t4(const PartialParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemPartial &sm = *reinterpret_cast<SmemPartial *>(smem_raw);
  const int split = blockIdx.x;
  const int unit = blockIdx.y;
  const int hg = unit % p.n_hg;
  const int bk = unit / p.n_hg;  // b * Hkv + kv-head
  const int b = bk / p.Hkv, kvh = bk % p.Hkv;
  int Lb = p.L;
  if (p.seq_lens) {
    int v = p.seq_lens[b];
    if (v < 1 || v > p.L) {
      if (threadIdx.x == 0) atomicExch(p.status, (int32_t)DEVERR_SEQLEN);
      v = v < 1 ? 1 : p.L;
    }
    Lb = v;
  }
  const int key0 = split * p.chunk;
  const int nkeys = max(0, min(key0 + p.chunk, Lb) - key0);
  const int ntiles = (nkeys + TILE - 1) / TILE;
  const int G = min(8, p.gq - hg * 8);
  const size_t unit_row0 = (size_t)bk * p.L;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], CWARPS);
    }
    sm.abort_flag = 0;
    sm.first_unconsumed = ntiles;
    sm.issued = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  float O[16][4];
  float M = -INFINITY, lsum = 0.f;
#pragma unroll
  for (int n = 0; n < 16; ++n) O[n][0] = O[n][1] = O[n][2] = O[n][3] = 0.f;

  if (warp == CWARPS) {
    // ---------------- producer: one elected lane streams K and V tiles
    if (lane == 0) {
      int i = 0;
      for (; i < ntiles; ++i) {
        const int s = i % NSTAGE;
        if (i >= NSTAGE && !mbar_wait_bounded(&sm.empty[s], ((i / NSTAGE) - 1) & 1, WAIT_LIMIT_NS)) {
          atomicExch(&sm.abort_flag, 1);
          atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
          break;
        }
        const int kf = key0 + i * TILE;
        const int nk = min(TILE, nkeys - i * TILE);
        const size_t start = (unit_row0 + kf) * T4_ROW;
        const size_t a0 = start & ~(size_t)15;
        const size_t a1 = (start + (size_t)nk * T4_ROW + 15) & ~(size_t)15;
        const uint32_t bytes = (uint32_t)(a1 - a0);
        mbar_arrive_expect_tx(&sm.full[s], 2 * bytes);
        bulk_g2s(sm.kbuf[s], p.kc + a0, bytes, &sm.full[s]);
        bulk_g2s(sm.vbuf[s], p.vc + a0, bytes, &sm.full[s]);
      }
      sm.issued = i;
    }
  } else {
    // ---------------- consumers
    const int hq = kvh * p.gq + hg * 8 + g;
    const bool head_ok = g < G;
    uint32_t qa[8][4];
    float qs = 0.f;
    if (head_ok) {
      const uint4 *qp = reinterpret_cast<const uint4 *>(p.qhl + (size_t)(b * p.Hq + hq) * 256);
      uint32_t hw[16], lw[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 a = qp[4 * t + i];        // hi words 16t .. 16t+15
        const uint4 c = qp[16 + 4 * t + i];   // lo words 64 + 16t ..
        hw[4 * i] = a.x, hw[4 * i + 1] = a.y, hw[4 * i + 2] = a.z, hw[4 * i + 3] = a.w;
        lw[4 * i] = c.x, lw[4 * i + 1] = c.y, lw[4 * i + 2] = c.z, lw[4 * i + 3] = c.w;
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[kk][0] = hw[2 * kk];
        qa[kk][1] = lw[2 * kk];
        qa[kk][2] = hw[2 * kk + 1];
        qa[kk][3] = lw[2 * kk + 1];
      }
      qs = p.qsc[2 * (b * p.Hq + hq)];
    } else {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) qa[kk][0] = qa[kk][1] = qa[kk][2] = qa[kk][3] = 0u;
    }
    const uint32_t klo[2] = {p.klo[0], p.klo[1]}, khi[2] = {p.khi[0], p.khi[1]};
    const uint32_t vlo[2] = {p.vlo[0], p.vlo[1]}, vhi[2] = {p.vhi[0], p.vhi[1]};
    const int kb = warp * 16;

    for (int i = 0; i < ntiles; ++i) {
      const int s = i % NSTAGE;
      if (!mbar_wait_bounded(&sm.full[s], (i / NSTAGE) & 1, WAIT_LIMIT_NS)) {
        atomicExch(&sm.abort_flag, 1);
        atomicMin(&sm.first_unconsumed, i);
        if (lane == 0) atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
        break;
      }
      const int kf = key0 + i * TILE;
      const int nk = min(TILE, nkeys - i * TILE);
      const size_t start = (unit_row0 + kf) * T4_ROW;
      const uint8_t *Ks = sm.kbuf[s] + (start & 15);
      const uint8_t *Vs = sm.vbuf[s] + (start & 15);
      if (kb < nk) {
        // ---- scores: two n-tiles of 8 keys (kb + g and kb + 8 + g for this lane)
        float sc0[4] = {0.f, 0.f, 0.f, 0.f}, sc1[4] = {0.f, 0.f, 0.f, 0.f};
        const uint8_t *kp0 = Ks + (kb + g) * T4_ROW + 4 + 16 * t;
        const uint8_t *kp1 = kp0 + 8 * T4_ROW;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t r[4];
          decode8<0x5140u, 0x7362u>(*reinterpret_cast<const uint32_t *>(kp0 + 4 * w), klo, khi, r);
          mma_f16(sc0, qa[2 * w], r[0], r[1]);
          mma_f16(sc0, qa[2 * w + 1], r[2], r[3]);
          decode8<0x5140u, 0x7362u>(*reinterpret_cast<const uint32_t *>(kp1 + 4 * w), klo, khi, r);
          mma_f16(sc1, qa[2 * w], r[0], r[1]);
          mma_f16(sc1, qa[2 * w + 1], r[2], r[3]);
        }
        // ---- online softmax over this lane's 4 keys of head g
        const int kl[4] = {kb + 2 * t, kb + 2 * t + 1, kb + 8 + 2 * t, kb + 9 + 2 * t};
        float sv[4] = {sc0[0] + sc0[2], sc0[1] + sc0[3], sc1[0] + sc1[2], sc1[1] + sc1[3]};
        float uv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float nkn = *reinterpret_cast<const float *>(Ks + kl[e] * T4_ROW);
          const float nvn = *reinterpret_cast<const float *>(Vs + kl[e] * T4_ROW);
          const bool valid = kl[e] < nk;
          sv[e] = valid ? sv[e] * (nkn * qs) : -INFINITY;
          uv[e] = valid ? sv[e] + fmaxf(log2_approx(nvn), -64.f) : -INFINITY;
          if (SCORES && valid && head_ok)
            p.scores[((size_t)(b * p.Hq + hq)) * p.L + kf + kl[e]] = sv[e] * LN2;
        }
        float bm = fmaxf(fmaxf(uv[0], uv[1]), fmaxf(uv[2], uv[3]));
        bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 2));
        if (bm > M) {
          const float alpha = exp2_approx(M - bm);
          M = bm;
          lsum *= alpha;
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            O[n][0] *= alpha, O[n][1] *= alpha, O[n][2] *= alpha, O[n][3] *= alpha;
          }
        }
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float pp[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          lsum += exp2_approx(sv[e] - Mu);
          pp[e] = exp2_approx(uv[e] - Mu + P_SHIFT);
        }
        uint32_t pa[4];
        split_half2(pp[0], pp[1], pa[0], pa[1]);
        split_half2(pp[2], pp[3], pa[2], pa[3]);
        // ---- PV: V_hat columns 16 g + n of keys 2t, 2t+1 (b0b1) and 2t+8, 2t+9 (b2b3)
        const uint8_t *v0 = Vs + (kb + 2 * t) * T4_ROW + 4 + 8 * g;
        const uint8_t *v2 = v0 + 8 * T4_ROW;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t xa = *reinterpret_cast<const uint32_t *>(v0 + 4 * half);
          const uint32_t xb = *reinterpret_cast<const uint32_t *>(v0 + T4_ROW + 4 * half);
          const uint32_t xc = *reinterpret_cast<const uint32_t *>(v2 + 4 * half);
          const uint32_t xd = *reinterpret_cast<const uint32_t *>(v2 + T4_ROW + 4 * half);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint32_t sel = q ? 0x7362u : 0x5140u;
            uint32_t r01[4], r23[4];
            decode8<0x6240u, 0x7351u>(prmt(xa, xb, sel), vlo, vhi, r01);
            decode8<0x6240u, 0x7351u>(prmt(xc, xd, sel), vlo, vhi, r23);
#pragma unroll
            for (int dd = 0; dd < 4; ++dd) mma_f16(O[half * 8 + q * 4 + dd], pa, r01[dd], r23[dd]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
    }
    lsum += __shfl_xor_sync(FULL_MASK, lsum, 1);
    lsum += __shfl_xor_sync(FULL_MASK, lsum, 2);
  }

  // ---------------- merge the consumer warps' states, write this split's partial
  __syncthreads();
  if (warp < CWARPS && t == 0) {
    sm.mw[warp][g] = M;
    sm.lw[warp][g] = lsum;
  }
  __syncthreads();
  float fac = 0.f;
  if (warp < CWARPS) {
    float ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < CWARPS; ++w) ms = fmaxf(ms, sm.mw[w][g]);
    fac = (M == -INFINITY) ? 0.f : exp2_approx(M - ms);
  }
  for (int w = 0; w < CWARPS; ++w) {
    if (warp == w && g < G) {
      float *orow = sm.osm[g];
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const float a = (O[n][0] + O[n][2]) * fac, c = (O[n][1] + O[n][3]) * fac;
        if (w == 0) {
          orow[32 * t + n] = a;
          orow[32 * t + 16 + n] = c;
        } else {
          orow[32 * t + n] += a;
          orow[32 * t + 16 + n] += c;
        }
      }
    }
    __syncthreads();
  }
  for (int idx = threadIdx.x; idx < G * (D + 6); idx += NTHREADS) {
    const int gg = idx / (D + 6), j = idx % (D + 6);
    const int hq = kvh * p.gq + hg * 8 + gg;
    float *dst = p.part + ((size_t)(b * p.Hq + hq) * p.n_split + split) * PARTIAL_FLOATS;
    float ms = -INFINITY;
    for (int w = 0; w < CWARPS; ++w) ms = fmaxf(ms, sm.mw[w][gg]);
    if (j == 0) {
      dst[0] = ms;
    } else if (j == 1) {
      float ls = 0.f;
      if (ms != -INFINITY)
        for (int w = 0; w < CWARPS; ++w)
          if (sm.mw[w][gg] != -INFINITY) ls += sm.lw[w][gg] * exp2_approx(sm.mw[w][gg] - ms);
      dst[1] = ls;
    } else if (j < 6) {
      dst[j] = 0.f;
    } else {
      dst[j] = (ms == -INFINITY) ? 0.f : sm.osm[gg][j - 6];
    }
  }
  // drain: if a wait gave up, let every issued copy land before the CTA exits
  if (threadIdx.x == 0 && sm.abort_flag) {
    for (int i = sm.first_unconsumed; i < sm.issued; ++i)
      (void)mbar_wait_bounded(&sm.full[i % NSTAGE], (i / NSTAGE) & 1, WAIT_LIMIT_NS);
  }
}

struct CombineParams {
  const float *part;
  int n_split;
  const float *r;   // R (row-major) of the value rotation, or null
  float inv_vscale; // 1 / (2^14 * alpha_V)
  float *out;
};

__global__ void __launch_bounds__(D) k_combine(const CombineParams p) {
  __shared__ float o[D];
  const int bh = blockIdx.x, j = threadIdx.x;
  const float *part = p.part + (size_t)bh * p.n_split * PARTIAL_FLOATS;
  float ms = -INFINITY;
  for (int s = 0; s < p.n_split; ++s)
    if (part[s * PARTIAL_FLOATS + 1] > 0.f) ms = fmaxf(ms, part[s * PARTIAL_FLOATS]);
  float lsum = 0.f, acc = 0.f;
  for (int s = 0; s < p.n_split; ++s) {
    const float *ps = part + s * PARTIAL_FLOATS;
    if (ps[1] > 0.f) {
      const float w = exp2f(ps[0] - ms);
      lsum += w * ps[1];
      acc += w * ps[6 + j];
    }
  }
  o[j] = acc * p.inv_vscale / lsum;
  __syncthreads();
  float r = o[j];
  if (p.r) {
    r = 0.f;
    for (int k = 0; k < D; ++k) r = fmaf(p.r[k * D + j], o[k], r);  // (R^T o)_j
  }
  p.out[(size_t)bh * D + j] = r;
}

}  // namespace

bool decode_shape(const tq_ctx *k, const tq_ctx *v, int B, int Hq, int Hkv, int L,
                  DecodeShape *s) {
  (void)v;
  s->B = B, s->Hq = Hq, s->Hkv = Hkv, s->L = L;
  s->gq = Hq / Hkv;
  s->n_hg = (s->gq + 7) / 8;
  const int units = B * Hkv * s->n_hg;
  const int slots = k->num_sms * 2;
  int want = (4 * slots + units - 1) / units;
  if (want < 1) want = 1;
  int max_split = (L + 255) / 256;
  if (max_split < 1) max_split = 1;
  int n = want < max_split ? want : max_split;
  int chunk = (L + n - 1) / n;
  chunk = (chunk + TILE - 1) / TILE * TILE;
  s->chunk = chunk;
  s->n_split = (L + chunk - 1) / chunk;
  return true;
}

Workspace carve_workspace(const DecodeShape &s, void *base) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t nq = (size_t)s.B * s.Hq;
  const size_t b_qhl = up(nq * 256 * sizeof(uint32_t));
  const size_t b_qsc = up(nq * 2 * sizeof(float));
  const size_t b_part = up(nq * s.n_split * PARTIAL_FLOATS * sizeof(float));
  Workspace w{};
  uint8_t *p = static_cast<uint8_t *>(base);
  w.qhl = reinterpret_cast<uint32_t *>(p);
  w.qsc = reinterpret_cast<float *>(p ? p + b_qhl : nullptr);
  w.partials = reinterpret_cast<float *>(p ? p + b_qhl + b_qsc : nullptr);
  w.bytes = b_qhl + b_qsc + b_part;
  return w;
}

cudaError_t launch_prepare_q(const tq_ctx *k, const void *q, int q_dtype, const DecodeShape &s,
                             float scale, const Workspace &ws, cudaStream_t st) {
  QprepParams p{};
  p.q = q;
  p.q_dtype = q_dtype;
  p.n_q = s.B * s.Hq;
  p.rt = k->d_pit;
  p.mul = LOG2E * scale / k->f16.alpha;
  p.qhl = ws.qhl;
  p.qsc = ws.qsc;
  const int grid = (p.n_q + QWARPS - 1) / QWARPS;
  k_prepare_q<<<grid, QWARPS * 32, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_partial(const tq_ctx *k, const tq_ctx *v, const uint8_t *kc,
                           const uint8_t *vc, const int32_t *seq_lens, const DecodeShape &s,
                           float *scores_dbg, const Workspace &ws, cudaStream_t st) {
  PartialParams p{};
  p.kc = kc, p.vc = vc, p.seq_lens = seq_lens;
  p.B = s.B, p.Hq = s.Hq, p.Hkv = s.Hkv, p.L = s.L, p.gq = s.gq, p.n_hg = s.n_hg;
  p.n_split = s.n_split, p.chunk = s.chunk;
  p.qhl = ws.qhl, p.qsc = ws.qsc, p.part = ws.partials, p.scores = scores_dbg;
  for (int i = 0; i < 2; ++i) {
    p.klo[i] = k->f16.lo[i], p.khi[i] = k->f16.hi[i];
    p.vlo[i] = v->f16.lo[i], p.vhi[i] = v->f16.hi[i];
  }
  p.status = k->d_status;
  const size_t smem = sizeof(SmemPartial);
  dim3 grid(s.n_split, s.B * s.Hkv * s.n_hg);
  cudaError_t e;
  if (scores_dbg) {
    e = cudaFuncSetAttribute(k_partial_t4<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_partial_t4<true><<<grid, NTHREADS, smem, st>>>(p);
  } else {
    e = cudaFuncSetAttribute(k_partial_t4<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_partial_t4<false><<<grid, NTHREADS, smem, st>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const tq_ctx *k, const tq_ctx *v, const DecodeShape &s, float *out,
                           const Workspace &ws, cudaStream_t st) {
  (void)k;
  CombineParams p{};
  p.part = ws.partials;
  p.n_split = s.n_split;
  p.r = v->d_pi;
  p.inv_vscale = 1.0f / (exp2f(P_SHIFT) * v->f16.alpha);
  p.out = out;
  k_combine<<<s.B * s.Hq, D, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tq
