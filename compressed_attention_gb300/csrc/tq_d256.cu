// Head dimension 256 (turbo4 keys and values), the per-head-dimension case of
// "turboquant_plus: how the turbo4 KV format came back", section 9: a 256-element row is
// rotated as a whole (randomized Hadamard of order 256 or a dense 256 x 256 Pi), quantized
// with the 16-level codebook of N(0, 1/256), and stored as two consecutive 68-byte turbo4
// blocks (the format's 128-element block: fp32 norm + qs[64]); block c holds elements
// 128c .. 128c+127 of the rotated row and the row's norm.  Readers scale each block by its
// own stored norm.
//
// Kernels:
//   k_write_d256    SET_ROWS, lane l of a warp holding elements 8l .. 8l+7 (the canonical
//                   norm tree: a balanced pairwise sum in the lane, then the butterfly over
//                   the lanes; IEEE division).  Randomized Hadamard: one warp per row, the
//                   butterfly with stages 1, 2, 4 in the lane and 8 .. 128 across lanes,
//                   x 1/16.  Dense Pi: one CTA per row, the 256 x 256 product split over
//                   its eight warps (32 rows of R^T each, summed in shared memory).
//   k_dequant_d256  reconstruction, one warp per row.
//   k_prepare_q256  q_rot = R q (one CTA per query, the product split as above), scaled
//                   and split into fp16 hi + lo operands.
//   k_partial_d256  split-K decode: CTA (unit, split) of four warps, each taking 16 keys at
//                   a time; scores and PV as m16n8k16 MMAs with table-decoded fp16
//                   centroids, per-block norms on the scores, the largest value norm in the
//                   softmax exponent and each block's ratio to it in that block's
//                   probability operand.
//   k_combine_d256  merge of the splits (one CTA per head, the splits shared by its warps)
//                   and the un-rotation R^T o (the product split as above).
#include <cuda_fp16.h>
#include <math.h>

#include "tq_decode_common.cuh"
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int WARPS2 = 8;          // warps per CTA of the write, dequantize and q kernels
constexpr int PW = 4;              // warps per CTA of the split-K kernel
constexpr int PSTAGE = 16 * ROW256;  // one warp's 16 rows of one tensor (2176 B)

// Canonical norm of the row, lane l holding elements 8l .. 8l+7: the lane's squares summed
// as ((x0^2 + x1^2) + (x2^2 + x3^2)) + ((x4^2 + x5^2) + (x6^2 + x7^2)), then the butterfly
// over the lanes at distances 16, 8, 4, 2, 1 (every lane ends with the same value).
__device__ __forceinline__ float norm256(const float (&x)[8]) {
  float s[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] = __fadd_rn(__fmul_rn(x[2 * i], x[2 * i]), __fmul_rn(x[2 * i + 1], x[2 * i + 1]));
  float p = __fadd_rn(__fadd_rn(s[0], s[1]), __fadd_rn(s[2], s[3]));
#pragma unroll
  for (int h = 16; h >= 1; h >>= 1) p = __fadd_rn(p, __shfl_xor_sync(FULL_MASK, p, h));
  return __fsqrt_rn(p);
}

__device__ __forceinline__ void load8(const void *src, int dtype, int64_t row, int64_t stride, int lane,
                                      float (&x)[8]) {
  if (dtype == TQ_DTYPE_F32) {
    const float4 *s = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + row * stride + 8 * lane);
    const float4 a = s[0], b = s[1];
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
  } else {
    const uint2 *s = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(src) + row * stride + 8 * lane);
    const uint2 a = s[0], b = s[1];
    const uint32_t w[4] = {a.x, a.y, b.x, b.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) x[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu), x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
}

struct Write256 {
  const void *src;
  int src_dtype;
  int64_t n_rows, stride;
  const int64_t *row_ids;
  uint8_t *dst;
  int64_t dst_rows;
  int32_t *status;
  const float *rt;    // dense: R^T fp32 [256][256]
  uint32_t neg[8];    // WHT: bit j set when sign j is -1
  float b[15];        // decision boundaries
};

// #{k : y > b_k} over the 15 boundaries (strict: ties to the lower index).
__device__ __forceinline__ uint32_t count_below(float y, const float *b) {
  uint32_t n = 0;
#pragma unroll
  for (int k = 0; k < 15; ++k) n += (y > b[k]) ? 1u : 0u;
  return n;
}

// y = M^T x for a 256 x 256 fp32 matrix (row k at mt + 256 k) and x in shared memory, by
// the CTA's eight warps: warp w sums rows 32w .. 32w+31 (their loads issued eight rows at a
// time), lane l outputs 8l .. 8l+7; the slices meet in red[8][256] and every warp sums them
// in warp order.  Ends with a barrier after which red and x may be rewritten only after
// another barrier.
__device__ __forceinline__ void cta_matvec256(const float *mt, const float *xs, float (*red)[D256], int warp,
                                              int lane, float (&y)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll 8
  for (int i = 0; i < 32; ++i) {
    const int k = 32 * warp + i;
    const float xk = xs[k];
    const float4 *r4 = reinterpret_cast<const float4 *>(mt + (size_t)k * D256 + 8 * lane);
    const float4 a = __ldg(r4), b = __ldg(r4 + 1);
    y[0] = fmaf(a.x, xk, y[0]), y[1] = fmaf(a.y, xk, y[1]), y[2] = fmaf(a.z, xk, y[2]), y[3] = fmaf(a.w, xk, y[3]);
    y[4] = fmaf(b.x, xk, y[4]), y[5] = fmaf(b.y, xk, y[5]), y[6] = fmaf(b.z, xk, y[6]), y[7] = fmaf(b.w, xk, y[7]);
  }
  float4 *r4 = reinterpret_cast<float4 *>(&red[warp][8 * lane]);
  r4[0] = make_float4(y[0], y[1], y[2], y[3]);
  r4[1] = make_float4(y[4], y[5], y[6], y[7]);
  __syncthreads();
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll
  for (int w = 0; w < WARPS2; ++w) {
    const float4 *q4 = reinterpret_cast<const float4 *>(&red[w][8 * lane]);
    const float4 a = q4[0], b = q4[1];
    y[0] += a.x, y[1] += a.y, y[2] += a.z, y[3] += a.w, y[4] += b.x, y[5] += b.y, y[6] += b.z, y[7] += b.w;
  }
}

template <int SRC, bool DENSE>
__global__ void __launch_bounds__(WARPS2 * 32) k_write_d256(const Write256 p) {
  __shared__ float sb[16];
  pdl_trigger();
  if (threadIdx.x < 15) sb[threadIdx.x] = p.b[threadIdx.x];
  __syncthreads();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (DENSE) {
    // one CTA per row: warp 0 normalises it, the eight warps share the rotation, warp 0
    // quantizes and packs
    __shared__ __align__(16) float us[D256];
    __shared__ __align__(16) float red[WARPS2][D256];
    __shared__ float nsh;
    for (int64_t row = blockIdx.x; row < p.n_rows; row += gridDim.x) {
      const int64_t slot = p.row_ids ? p.row_ids[row] : row;  // the same for the whole CTA
      if (slot < 0 || slot >= p.dst_rows) {
        if (threadIdx.x == 0) atomicExch(p.status, (int32_t)DEVERR_ROW_OOB);
        continue;
      }
      if (warp == 0) {
        float v[8];
        load8(p.src, SRC, row, p.stride, lane, v);
        const float n = norm256(v);
#pragma unroll
        for (int e = 0; e < 8; ++e) us[8 * lane + e] = (n == 0.0f) ? 0.0f : __fdiv_rn(v[e], n);
        if (lane == 0) nsh = n;
      }
      __syncthreads();
      float y[8];
      cta_matvec256(p.rt, us, red, warp, lane, y);
      if (warp == 0) {
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) word |= count_below(y[e], sb) << (4 * e);
        uint8_t *blk = p.dst + slot * ROW256 + 68 * (lane >> 4);
        reinterpret_cast<uint32_t *>(blk + 4)[lane & 15] = word;
        if ((lane & 15) == 0) *reinterpret_cast<float *>(blk) = nsh;
      }
      __syncthreads();  // us, red and nsh free for the next row
    }
    return;
  }
  for (int64_t row = (int64_t)blockIdx.x * WARPS2 + warp; row < p.n_rows; row += (int64_t)gridDim.x * WARPS2) {
    const int64_t slot = p.row_ids ? p.row_ids[row] : row;
    if (slot < 0 || slot >= p.dst_rows) {
      if (lane == 0) atomicExch(p.status, (int32_t)DEVERR_ROW_OOB);
      continue;
    }
    float v[8];
    load8(p.src, SRC, row, p.stride, lane, v);
    const float n = norm256(v);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = (n == 0.0f) ? 0.0f : __fdiv_rn(v[e], n);
    float y[8];
    {
      // signs (exact), the butterfly stages h = 1, 2, 4 in the lane, 8 .. 128 across lanes
      // (the lower element of a pair keeps a + b, the upper a - b), then x RN(1/16) = 1/16
      const uint32_t sw = p.neg[lane >> 2] >> (8 * (lane & 3));
#pragma unroll
      for (int e = 0; e < 8; ++e)
        v[e] = __uint_as_float(__float_as_uint(v[e]) ^ (((sw >> e) & 1u) << 31));
#pragma unroll
      for (int h = 1; h <= 4; h <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (!(e & h)) {
            const float a = v[e], b = v[e + h];
            v[e] = __fadd_rn(a, b);
            v[e + h] = __fsub_rn(a, b);
          }
#pragma unroll
      for (int m = 1; m <= 16; m <<= 1) {
        const bool upper = lane & m;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float o = __shfl_xor_sync(FULL_MASK, v[e], m);
          v[e] = upper ? __fsub_rn(o, v[e]) : __fadd_rn(v[e], o);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(v[e], 0.0625f);
    }
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) word |= count_below(y[e], sb) << (4 * e);
    uint8_t *blk = p.dst + slot * ROW256 + 68 * (lane >> 4);
    reinterpret_cast<uint32_t *>(blk + 4)[lane & 15] = word;
    if ((lane & 15) == 0) *reinterpret_cast<float *>(blk) = n;
  }
}

struct Dequant256 {
  const uint8_t *cache;
  int64_t n_rows;
  int unrotate;
  const float *r;  // R fp32 [256][256], row-major
  float c[16];
  float *dst;
};

__global__ void __launch_bounds__(WARPS2 * 32) k_dequant_d256(const Dequant256 p) {
  __shared__ float cs[16];
  if (threadIdx.x < 16) cs[threadIdx.x] = p.c[threadIdx.x];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t row = (int64_t)blockIdx.x * WARPS2 + warp; row < p.n_rows; row += (int64_t)gridDim.x * WARPS2) {
    const uint8_t *blk = p.cache + row * ROW256 + 68 * (lane >> 4);
    const float n = *reinterpret_cast<const float *>(blk);
    const uint32_t word = reinterpret_cast<const uint32_t *>(blk + 4)[lane & 15];
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = n * cs[(word >> (4 * e)) & 15u];
    float x[8];
    if (p.unrotate) {
      // x_j = sum_k R[k][j] y_k: lane l takes j = 8l .. 8l+7 from row k of R
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.f;
#pragma unroll 16
      for (int k = 0; k < D256; ++k) {
        const float yk = __shfl_sync(FULL_MASK, y[k & 7], k >> 3);
        const float4 *r4 = reinterpret_cast<const float4 *>(p.r + (size_t)k * D256 + 8 * lane);
        const float4 a = r4[0], b = r4[1];
        x[0] = fmaf(a.x, yk, x[0]), x[1] = fmaf(a.y, yk, x[1]), x[2] = fmaf(a.z, yk, x[2]), x[3] = fmaf(a.w, yk, x[3]);
        x[4] = fmaf(b.x, yk, x[4]), x[5] = fmaf(b.y, yk, x[5]), x[6] = fmaf(b.z, yk, x[6]), x[7] = fmaf(b.w, yk, x[7]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = y[e];
    }
    float4 *o4 = reinterpret_cast<float4 *>(p.dst + row * D256 + 8 * lane);
    o4[0] = make_float4(x[0], x[1], x[2], x[3]);
    o4[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
}

struct Prep256 {
  const void *q;
  int q_dtype;
  int n_q;
  const float *rt;  // R^T fp32 [256][256]
  float mul;        // log2(e) * scale / alpha_K
  uint32_t *qhl;    // [n_q][256]: fp16 hi of q_rot[0..255], then fp16 lo
  float *qsc;       // [n_q][2]
};

__global__ void __launch_bounds__(WARPS2 * 32) k_prepare_q256(const Prep256 p) {
  // one CTA per query: warp 0 loads it, the eight warps share q_rot = R q, warp 0 splits
  __shared__ __align__(16) float xs[D256];
  __shared__ __align__(16) float red[WARPS2][D256];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qi = blockIdx.x;
  if (qi >= p.n_q) return;
  if (warp == 0) {
    float x[8];
    if (p.q_dtype == TQ_DTYPE_F32) {
      load8(p.q, TQ_DTYPE_F32, qi, D256, lane, x);
    } else if (p.q_dtype == TQ_DTYPE_BF16) {
      load8(p.q, TQ_DTYPE_BF16, qi, D256, lane, x);
    } else {
      const uint4 w = reinterpret_cast<const uint4 *>(static_cast<const __half *>(p.q) + (size_t)qi * D256)[lane];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ws[i]));
        x[2 * i] = f.x, x[2 * i + 1] = f.y;
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) xs[8 * lane + e] = x[e];
  }
  __syncthreads();
  float y[8];
  cta_matvec256(p.rt, xs, red, warp, lane, y);
  if (warp != 0) return;
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    y[e] *= p.mul;
    amax = fmaxf(amax, fabsf(y[e]));
  }
#pragma unroll
  for (int h = 16; h >= 1; h >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, h));
  int ex = 0;
  if (amax > 0.f && isfinite(amax)) ex = ilogbf(amax) - 13;
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = ldexpf(y[2 * i], -ex), b = ldexpf(y[2 * i + 1], -ex);
    split_half2(a, b, hi[i], lo[i]);
  }
  uint32_t *dst = p.qhl + (size_t)qi * 256;
  reinterpret_cast<uint4 *>(dst)[lane] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  reinterpret_cast<uint4 *>(dst + 128)[lane] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  if (lane == 0) {
    p.qsc[2 * qi] = ldexpf(1.0f, ex);
    p.qsc[2 * qi + 1] = 0.f;
  }
}

struct Part256 {
  const uint8_t *kc, *vc;
  const int32_t *seq_lens;
  int B, Hq, Hkv, L, gq, n_hg, n_split, chunk;
  const uint32_t *qhl;
  const float *qsc;
  float *part;  // [B*Hq][n_split][PARTIAL256]: max, sum, 6 spare, acc[256] (16-byte aligned)
  uint32_t kc16[8], vc16[8];
  int32_t *status;
};

// Shared memory: the decode table lut[b][s] (s < 32 key slots, 32.. value slots: entry =
// (c[b & 15], c[b >> 4]) fp16x2 of the key or value table; lane l reads slot l or 32 + l, so
// a warp's 32 lookups hit 32 banks), each warp's 16 K and 16 V rows, the merge scratch.
struct Smem256 {
  uint32_t lut[256][64];
  union {
    uint8_t kv[PW][2][2][PSTAGE];  // warp, buffer (double-buffered), K / V
    float osm[PW][4][D256];        // the merge scratch, after the last block
  };
  float mw[PW][4], lw[PW][4];
};

// Start copying a warp's block of nk rows (keys kb ..) of K and V into shared memory
// (8-byte pieces of the valid rows; rows start 8-byte aligned), as one cp.async group.
__device__ __forceinline__ void stage_block(uint8_t *ks, uint8_t *vs, const uint8_t *kc, const uint8_t *vc,
                                            size_t row0, int nk, int lane) {
  const int n8 = nk * (ROW256 / 8);
  const uint8_t *kg = kc + row0 * ROW256, *vg = vc + row0 * ROW256;
  for (int i = lane; i < n8; i += 32) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(ks + 8 * i)), "l"(kg + 8 * i) : "memory");
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(vs + 8 * i)), "l"(vg + 8 * i) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ uint32_t lut_at(const uint32_t *lut, uint32_t laneword, uint32_t w, int i) {
  return lut[((w >> (8 * i)) & 0xFFu) * 64 + laneword];
}

// Physical key (of 16) of score row r, and the B-operand key order, as in the turbo4
// split-K kernel: rows g and g+8 of lane group g; the PV operand of lane (g, t) takes keys
// a_t, a_t+2, a_t+4, a_t+6 with a_t = {0, 1, 8, 9}[t].
__device__ __forceinline__ int key_row(int r) {
  return ((r & 1) | ((r & 2) << 2) | ((r & 4) >> 1) | ((r & 8) >> 1));
}

__global__ void __launch_bounds__(PW * 32, 1) k_partial_d256(const Part256 p) {
  extern __shared__ __align__(16) uint8_t smem2[];
  Smem256 &sm = *reinterpret_cast<Smem256 *>(smem2);
  pdl_trigger();
  for (int piece = threadIdx.x; piece < 256 * 64; piece += PW * 32) {
    const int byte = piece >> 6, slot = piece & 63;
    const uint32_t *c16 = slot >= 32 ? p.vc16 : p.kc16;
    const uint32_t lo = (c16[(byte & 15) >> 1] >> (16 * (byte & 1))) & 0xFFFFu;
    const uint32_t hi = (c16[(byte >> 4) >> 1] >> (16 * ((byte >> 4) & 1))) & 0xFFFFu;
    sm.lut[byte][slot] = lo | (hi << 16);
  }
  __syncthreads();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int unit = blockIdx.x / p.n_split, split = blockIdx.x % p.n_split;
  const int hg = unit % p.n_hg, bk = unit / p.n_hg;
  const int b = bk / p.Hkv, kvh = bk % p.Hkv;
  const int G = min(4, p.gq - hg * 4);
  const int head0 = kvh * p.gq + hg * 4;
  int Lb = p.L;
  if (p.seq_lens) {
    const int v = p.seq_lens[b];
    if ((v < 1 || v > p.L) && threadIdx.x == 0 && split == 0 && hg == 0 && kvh == 0)
      atomicExch(p.status, (int32_t)DEVERR_SEQLEN);
    Lb = v < 1 ? 1 : (v > p.L ? p.L : v);
  }
  const int k0 = split * p.chunk, k1 = min(Lb, k0 + p.chunk);
  const size_t unit_row0 = (size_t)bk * p.L;

  // q as the B operand: column g = (head slot g/2, fp16 hi (g even) or lo (g odd)); block
  // half hb, k-step s: dims 128 hb + 32 t + 4 s .. + 3 in lane t
  const int hs = g >> 1;
  uint32_t qb[2][8][2];
  float qs = 0.f;
  if (hs < G) {
    const uint32_t *qw = p.qhl + (size_t)(b * p.Hq + head0 + hs) * 256 + (g & 1) * 128 + 16 * t;
#pragma unroll
    for (int hb = 0; hb < 2; ++hb)
#pragma unroll
      for (int s = 0; s < 8; ++s) qb[hb][s][0] = qw[64 * hb + 2 * s], qb[hb][s][1] = qw[64 * hb + 2 * s + 1];
  } else {
#pragma unroll
    for (int hb = 0; hb < 2; ++hb)
#pragma unroll
      for (int s = 0; s < 8; ++s) qb[hb][s][0] = qb[hb][s][1] = 0u;
  }
  if (t < G) qs = p.qsc[2 * (b * p.Hq + head0 + t)];
  const int pk0 = key_row(g), pk1 = key_row(g + 8);
  const int at = (t & 1) | ((t & 2) << 2);
  const int src0 = 4 * t + hs, src1 = 4 * (4 + t) + hs;
  const float lo_sel = (g & 1) ? 1.f : 0.f;
  const uint32_t kword = lane, vword = 32 + lane;

  float O[16][4];
#pragma unroll
  for (int mt = 0; mt < 16; ++mt) O[mt][0] = O[mt][1] = O[mt][2] = O[mt][3] = 0.f;
  float M = -INFINITY, lsum = 0.f;
  // the warp's blocks of 16 keys: kb = k0 + 16 (warp + PW i); each block's K and V rows are
  // copied into one of two buffers while the previous block is computed
  int buf = 0;
  if (k0 + 16 * warp < k1)
    stage_block(sm.kv[warp][0][0], sm.kv[warp][0][1], p.kc, p.vc, unit_row0 + k0 + 16 * warp,
                min(16, k1 - k0 - 16 * warp), lane);
  for (int kb = k0 + 16 * warp; kb < k1; kb += 16 * PW, buf ^= 1) {
    const int nk = min(16, k1 - kb);
    const int kn = kb + 16 * PW;
    if (kn < k1) {
      stage_block(sm.kv[warp][buf ^ 1][0], sm.kv[warp][buf ^ 1][1], p.kc, p.vc, unit_row0 + kn, min(16, k1 - kn),
                  lane);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncwarp();
    const uint8_t *Ks = sm.kv[warp][buf][0], *Vs = sm.kv[warp][buf][1];
    const bool ok0 = pk0 < nk, ok1 = pk1 < nk;
    // ---- scores, block half by block half, each scaled by its own key norm
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sbb[4] = {0.f, 0.f, 0.f, 0.f};
      const uint8_t *kr0 = Ks + pk0 * ROW256 + 68 * hb + 4 + 16 * t;
      const uint8_t *kr1 = Ks + pk1 * ROW256 + 68 * hb + 4 + 16 * t;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t x0 = *reinterpret_cast<const uint32_t *>(kr0 + 4 * w);
        const uint32_t x1 = *reinterpret_cast<const uint32_t *>(kr1 + 4 * w);
        uint32_t d0[4], d1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) d0[i] = lut_at(&sm.lut[0][0], kword, x0, i), d1[i] = lut_at(&sm.lut[0][0], kword, x1, i);
        const uint32_t a0[4] = {d0[0], d1[0], d0[1], d1[1]};
        const uint32_t a1[4] = {d0[2], d1[2], d0[3], d1[3]};
        mma_f16(sa, a0, qb[hb][2 * w][0], qb[hb][2 * w][1]);
        mma_f16(sbb, a1, qb[hb][2 * w + 1][0], qb[hb][2 * w + 1][1]);
      }
      const float n0 = *reinterpret_cast<const float *>(Ks + pk0 * ROW256 + 68 * hb);
      const float n1 = *reinterpret_cast<const float *>(Ks + pk1 * ROW256 + 68 * hb);
      s0 = fmaf(n0, (sa[0] + sa[1]) + (sbb[0] + sbb[1]), s0);
      s1 = fmaf(n1, (sa[2] + sa[3]) + (sbb[2] + sbb[3]), s1);
    }
    s0 = ok0 ? s0 * qs : -INFINITY;
    s1 = ok1 ? s1 * qs : -INFINITY;
    // ---- values: the largest block norm in the exponent, each block's ratio to it in
    // that block's probability operand (rows past the valid keys: ratios 0)
    const float v00 = *reinterpret_cast<const float *>(Vs + pk0 * ROW256);
    const float v01 = *reinterpret_cast<const float *>(Vs + pk0 * ROW256 + 68);
    const float v10 = *reinterpret_cast<const float *>(Vs + pk1 * ROW256);
    const float v11 = *reinterpret_cast<const float *>(Vs + pk1 * ROW256 + 68);
    const float nv0 = fmaxf(v00, v01), nv1 = fmaxf(v10, v11);
    const float nu0 = ok0 ? fmaxf(log2_approx(nv0), -64.f) : 0.f;
    const float nu1 = ok1 ? fmaxf(log2_approx(nv1), -64.f) : 0.f;
    const float i0 = (ok0 && nv0 > 0.f) ? 1.f / nv0 : 0.f, i1 = (ok1 && nv1 > 0.f) ? 1.f / nv1 : 0.f;
    const float r00 = i0 > 0.f ? v00 * i0 : 0.f, r01 = i0 > 0.f ? v01 * i0 : 0.f;
    const float r10 = i1 > 0.f ? v10 * i1 : 0.f, r11 = i1 > 0.f ? v11 * i1 : 0.f;
    const float u0 = s0 + nu0, u1 = s1 + nu1;
    float bm = fmaxf(u0, u1);
    bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 4));
    bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 8));
    bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 16));
    if (bm > M + RESCALE_SLACK) {  // also taken while M is -inf
      const float alpha = exp2_approx(M - bm);
      M = bm;
      lsum *= alpha;
#pragma unroll
      for (int mt = 0; mt < 16; ++mt) O[mt][0] *= alpha, O[mt][1] *= alpha, O[mt][2] *= alpha, O[mt][3] *= alpha;
    }
    const float Mu = (M == -INFINITY) ? 0.f : M;
    lsum += exp2_approx(s0 - Mu) + exp2_approx(s1 - Mu);
    const float pp0 = exp2_approx(u0 - Mu + P_SHIFT), pp1 = exp2_approx(u1 - Mu + P_SHIFT);
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      // P^T as the B operand of block half hb (k 2t, 2t+1: keys a_t, a_t+2; k 2t+8, 2t+9:
      // keys a_t+4, a_t+6), gathered from the lanes that own those keys' scores
      const float q0 = pp0 * (hb ? r01 : r00), q1 = pp1 * (hb ? r11 : r10);
      const float va = __shfl_sync(FULL_MASK, q0, src0), vb = __shfl_sync(FULL_MASK, q0, src1);
      const float vc = __shfl_sync(FULL_MASK, q1, src0), vd = __shfl_sync(FULL_MASK, q1, src1);
      const __half2 hab = __floats2half2_rn(va, vb), hcd = __floats2half2_rn(vc, vd);
      const float2 fab = __half22float2(hab), fcd = __half22float2(hcd);
      const __half2 rab = __floats2half2_rn(fmaf(-lo_sel, fab.x, va), fmaf(-lo_sel, fab.y, vb));
      const __half2 rcd = __floats2half2_rn(fmaf(-lo_sel, fcd.x, vc), fmaf(-lo_sel, fcd.y, vd));
      const uint32_t pb0 = *reinterpret_cast<const uint32_t *>(&rab), pb1 = *reinterpret_cast<const uint32_t *>(&rcd);
      // O^T[dims x cols] += V_hat^T[dims x keys] P^T: lane (g, t) decodes bytes 8g .. 8g+7
      // of the block's qs for keys a_t + 2i
      const uint8_t *vp = Vs + at * ROW256 + 68 * hb + 4 + 8 * g;
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const uint32_t xa = *reinterpret_cast<const uint32_t *>(vp + 4 * w);
        const uint32_t xb = *reinterpret_cast<const uint32_t *>(vp + 2 * ROW256 + 4 * w);
        const uint32_t xc = *reinterpret_cast<const uint32_t *>(vp + 4 * ROW256 + 4 * w);
        const uint32_t xd = *reinterpret_cast<const uint32_t *>(vp + 6 * ROW256 + 4 * w);
        // byte i of zlo = (low nibble of key a, low nibble of key b) of byte 8g + 4w + i
        const uint32_t zlo_ab = (xa & 0x0F0F0F0Fu) | ((xb << 4) & 0xF0F0F0F0u);
        const uint32_t zhi_ab = ((xa >> 4) & 0x0F0F0F0Fu) | (xb & 0xF0F0F0F0u);
        const uint32_t zlo_cd = (xc & 0x0F0F0F0Fu) | ((xd << 4) & 0xF0F0F0F0u);
        const uint32_t zhi_cd = ((xc >> 4) & 0x0F0F0F0Fu) | (xd & 0xF0F0F0F0u);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint32_t a[4] = {lut_at(&sm.lut[0][0], vword, zlo_ab, jj), lut_at(&sm.lut[0][0], vword, zhi_ab, jj),
                                 lut_at(&sm.lut[0][0], vword, zlo_cd, jj), lut_at(&sm.lut[0][0], vword, zhi_cd, jj)};
          mma_f16(O[8 * hb + 4 * w + jj], a, pb0, pb1);
        }
      }
    }
    __syncwarp();  // every lane is done with this buffer before it is refilled
  }
  lsum += __shfl_xor_sync(FULL_MASK, lsum, 4);
  lsum += __shfl_xor_sync(FULL_MASK, lsum, 8);
  lsum += __shfl_xor_sync(FULL_MASK, lsum, 16);
  // ---- merge the four warps' states and write this split's partial of the unit's heads
  if (g == 0) sm.mw[warp][t] = M, sm.lw[warp][t] = lsum;
  __syncthreads();  // (also: every warp is done with the staging buffers the scratch reuses)
  float ms = -INFINITY;
#pragma unroll
  for (int w = 0; w < PW; ++w) ms = fmaxf(ms, sm.mw[w][t]);
  const float fac = (M == -INFINITY) ? 0.f : exp2_approx(M - ms);
  // rows g and g+8 of m-tile 8 hb + mt: dims 128 hb + 16 g + 2 mt and + 1
#pragma unroll
  for (int mt = 0; mt < 16; ++mt) {
    const int dm = 128 * (mt >> 3) + 16 * g + 2 * (mt & 7);
    sm.osm[warp][t][dm] = (O[mt][0] + O[mt][1]) * fac;
    sm.osm[warp][t][dm + 1] = (O[mt][2] + O[mt][3]) * fac;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D256; idx += PW * 32) {
    const int h = idx / D256, jd = idx % D256;
    float m2 = -INFINITY;
#pragma unroll
    for (int w = 0; w < PW; ++w) m2 = fmaxf(m2, sm.mw[w][h]);
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < PW; ++w) acc += sm.osm[w][h][jd];
    float *dst = p.part + ((size_t)(b * p.Hq + head0 + h) * p.n_split + split) * PARTIAL256;
    dst[ACC256 + jd] = (m2 == -INFINITY) ? 0.f : acc;
    if (jd < ACC256) {
      float v = 0.f;
      if (jd == 0) {
        v = m2;
      } else if (jd == 1 && m2 != -INFINITY) {
#pragma unroll
        for (int w = 0; w < PW; ++w)
          if (sm.mw[w][h] != -INFINITY) v += sm.lw[w][h] * exp2_approx(sm.mw[w][h] - m2);
      }
      dst[jd] = v;
    }
  }
}

struct Comb256 {
  const float *part;
  int n_heads, n_split;
  const float *r;  // R of the value rotation, fp32 [256][256] row-major
  float inv_vscale;
  float *out;
};

// One CTA per head: warp w merges splits w, w + 8, ... (m_w = max m_s, l_w, o_w with
// weights 2^(m_s - m_w)); the eight states meet in shared memory (m* = max m_w, l* = sum
// l_w 2^(m_w - m*), o = sum o_w 2^(m_w - m*) / l*, in the rotated basis); the eight warps
// then share out = R^T o.
__global__ void __launch_bounds__(WARPS2 * 32) k_combine_d256(const Comb256 p) {
  __shared__ __align__(16) float os[D256];
  __shared__ __align__(16) float red[WARPS2][D256];
  __shared__ float mws[WARPS2], lws[WARPS2];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  if (bh >= p.n_heads) return;
  const float *part = p.part + (size_t)bh * p.n_split * PARTIAL256;
  float ms = -INFINITY;
  for (int s = warp; s < p.n_split; s += WARPS2)
    if (part[(size_t)s * PARTIAL256 + 1] > 0.f) ms = fmaxf(ms, part[(size_t)s * PARTIAL256]);
  float l = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = warp; s < p.n_split; s += WARPS2) {
    const float *ps = part + (size_t)s * PARTIAL256;
    if (!(ps[1] > 0.f)) continue;
    const float w = exp2f(ps[0] - ms);
    l += w * ps[1];
    const float4 *a4 = reinterpret_cast<const float4 *>(ps + ACC256 + 8 * lane);
    const float4 a = a4[0], c = a4[1];
    o[0] = fmaf(w, a.x, o[0]), o[1] = fmaf(w, a.y, o[1]), o[2] = fmaf(w, a.z, o[2]), o[3] = fmaf(w, a.w, o[3]);
    o[4] = fmaf(w, c.x, o[4]), o[5] = fmaf(w, c.y, o[5]), o[6] = fmaf(w, c.z, o[6]), o[7] = fmaf(w, c.w, o[7]);
  }
  if (lane == 0) mws[warp] = ms, lws[warp] = l;
  float4 *r4 = reinterpret_cast<float4 *>(&red[warp][8 * lane]);
  r4[0] = make_float4(o[0], o[1], o[2], o[3]);
  r4[1] = make_float4(o[4], o[5], o[6], o[7]);
  __syncthreads();
  if (warp == 0) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS2; ++w) mx = fmaxf(mx, mws[w]);
    float lt = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < WARPS2; ++w) {
      if (mws[w] == -INFINITY) continue;
      const float f = exp2f(mws[w] - mx);
      lt += f * lws[w];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(f, red[w][8 * lane + e], acc[e]);
    }
    const float f = lt > 0.f ? p.inv_vscale / lt : 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) os[8 * lane + e] = acc[e] * f;
  }
  __syncthreads();
  float x[8];
  cta_matvec256(p.r, os, red, warp, lane, x);
  if (warp != 0) return;
  float4 *o4 = reinterpret_cast<float4 *>(p.out + (size_t)bh * D256 + 8 * lane);
  o4[0] = make_float4(x[0], x[1], x[2], x[3]);
  o4[1] = make_float4(x[4], x[5], x[6], x[7]);
}

int grid_rows(const tq_ctx *c, int64_t rows, int per_cta) {
  const int64_t want = (rows + per_cta - 1) / per_cta, cap = (int64_t)c->num_sms * 8;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_write_d256(const tq_ctx *ctx, const WriteLaunch &w, cudaStream_t st) {
  Write256 p{};
  p.src = w.src, p.src_dtype = w.src_dtype, p.n_rows = w.n_rows, p.stride = w.stride;
  p.row_ids = w.row_ids, p.dst = w.dst, p.dst_rows = w.dst_rows, p.status = ctx->d_status;
  p.rt = ctx->d_pit;
  for (int i = 0; i < 8; ++i) p.neg[i] = ctx->wht_neg[i];
  for (int k = 0; k < 15; ++k) p.b[k] = ctx->cb.b[k];
  const bool dense = ctx->p.rotation == TQ_ROT_DENSE, bf16 = w.src_dtype == TQ_DTYPE_BF16;
  // dense: one CTA per row (the rotation split over its warps); WHT: one warp per row
  const dim3 grid(grid_rows(ctx, w.n_rows, dense ? 1 : WARPS2)), block(WARPS2 * 32);
  if (dense)
    return bf16 ? launch_pdl(k_write_d256<TQ_DTYPE_BF16, true>, grid, block, 0, st, p)
                : launch_pdl(k_write_d256<TQ_DTYPE_F32, true>, grid, block, 0, st, p);
  return bf16 ? launch_pdl(k_write_d256<TQ_DTYPE_BF16, false>, grid, block, 0, st, p)
              : launch_pdl(k_write_d256<TQ_DTYPE_F32, false>, grid, block, 0, st, p);
}

cudaError_t launch_dequant_d256(const tq_ctx *ctx, const uint8_t *cache, int64_t n_rows, int unrotate,
                                float *dst, cudaStream_t st) {
  Dequant256 p{};
  p.cache = cache, p.n_rows = n_rows, p.unrotate = unrotate, p.r = ctx->d_pi, p.dst = dst;
  for (int k = 0; k < 16; ++k) p.c[k] = ctx->cb.c[k];
  k_dequant_d256<<<grid_rows(ctx, n_rows, WARPS2), WARPS2 * 32, 0, st>>>(p);
  return cudaGetLastError();
}

bool d256_shape(const tq_ctx *k, int B, int Hq, int Hkv, int L, D256Shape *s) {
  s->B = B, s->Hq = Hq, s->Hkv = Hkv, s->L = L;
  s->gq = Hq / Hkv;
  s->n_hg = (s->gq + 3) / 4;
  const int64_t units = (int64_t)B * Hkv * s->n_hg;
  // about four CTAs (two per SM) per SM's worth of work, 16-key blocks per split
  int64_t n_split = (4 * (int64_t)k->num_sms + units - 1) / units;
  const int64_t max_split = (L + 15) / 16;
  if (n_split > max_split) n_split = max_split;
  if (n_split < 1) n_split = 1;
  const int64_t per = (L + n_split - 1) / n_split;
  s->chunk = (int)(((per + 15) / 16) * 16);
  s->n_split = (int)((L + s->chunk - 1) / s->chunk);
  if (units * s->n_split > INT32_MAX || (int64_t)B * Hq * s->n_split * PARTIAL256 > ((int64_t)1 << 40)) return false;
  s->units = (int)units;
  return true;
}

size_t d256_workspace(const D256Shape &s, void *base, Workspace *w) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t nq = (size_t)s.B * s.Hq;
  const size_t b_qhl = up(nq * 256 * sizeof(uint32_t));
  const size_t b_qsc = up(nq * 2 * sizeof(float));
  const size_t b_part = up(nq * s.n_split * PARTIAL256 * sizeof(float));
  if (w) {
    *w = Workspace{};
    uint8_t *p = static_cast<uint8_t *>(base);
    w->qhl = reinterpret_cast<uint32_t *>(p);
    w->qsc = reinterpret_cast<float *>(p ? p + b_qhl : nullptr);
    w->partials = reinterpret_cast<float *>(p ? p + b_qhl + b_qsc : nullptr);
    w->bytes = b_qhl + b_qsc + b_part;
  }
  return b_qhl + b_qsc + b_part;
}

cudaError_t launch_prepare_q256(const tq_ctx *k, const void *q, int q_dtype, const D256Shape &s, float scale,
                                const Workspace &w, cudaStream_t st) {
  Prep256 p{};
  p.q = q, p.q_dtype = q_dtype, p.n_q = s.B * s.Hq, p.rt = k->d_pit;
  p.mul = LOG2E * scale / k->f16.alpha;
  p.qhl = w.qhl, p.qsc = w.qsc;
  return launch_pdl(k_prepare_q256, dim3(p.n_q), dim3(WARPS2 * 32), 0, st, p);
}

cudaError_t launch_partial_d256(const tq_ctx *k, const tq_ctx *v, const uint8_t *kc, const uint8_t *vc,
                                const int32_t *seq_lens, const D256Shape &s, const Workspace &w, cudaStream_t st) {
  Part256 p{};
  p.kc = kc, p.vc = vc, p.seq_lens = seq_lens;
  p.B = s.B, p.Hq = s.Hq, p.Hkv = s.Hkv, p.L = s.L, p.gq = s.gq, p.n_hg = s.n_hg;
  p.n_split = s.n_split, p.chunk = s.chunk;
  p.qhl = w.qhl, p.qsc = w.qsc, p.part = w.partials;
  for (int i = 0; i < 8; ++i) p.kc16[i] = k->f16.c16[i], p.vc16[i] = v->f16.c16[i];
  p.status = k->d_status;
  const size_t smem = sizeof(Smem256);
  cudaError_t e = kernel_smem_attr((const void *)k_partial_d256, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_partial_d256, dim3(s.units * s.n_split), dim3(PW * 32), smem, st, p);
}

cudaError_t launch_combine_d256(const tq_ctx *v, const D256Shape &s, float *out, const Workspace &w,
                                cudaStream_t st) {
  Comb256 p{};
  p.part = w.partials, p.n_heads = s.B * s.Hq, p.n_split = s.n_split, p.r = v->d_pi;
  p.inv_vscale = 1.0f / (exp2f(P_SHIFT) * v->f16.alpha);
  p.out = out;
  return launch_pdl(k_combine_d256, dim3(p.n_heads), dim3(WARPS2 * 32), 0, st, p);
}

}  // namespace tq
