// Write path / SET_ROWS kernels: norm -> normalise -> rotate -> nearest centroid
// -> pack, one warp per row ("turboquant_plus: how the turbo4 KV format came
// back", section 1 encode chain; section 2 dedicated SET_ROWS per format;
// sections 4-5 block layouts).  The V group quantizer follows "TurboQuant fused
// Triton kernels deep dive", "write path and codebook" (2-bit group
// quantization, value = code * scale + zero).
//
// The norm is the canonical fp32 tree: squares and adds rounded one by one (no
// contraction), sums of four consecutive squares, then pairwise combination over
// strides 16, 8, 4, 2, 1 of those 32 partial sums.  The WHT rotation is the
// butterfly of stages 1, 2, ..., 64 in that order, so its result is bit-identical
// to a plain sequential fp32 implementation of the same stage order.  The WHT
// kernel gives each of four threads four 8-element chunks of a row; the others give
// lane l of a warp elements 4l..4l+3 of its row and run the same trees across lanes.
#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_qprep.cuh"

namespace tq {

namespace {

constexpr int WARPS = 8;
constexpr int64_t SMALL_ROWS = 256;  // at most this many dense rows: one CTA per row
constexpr int ROWBUF = 72;  // per-warp staging for one packed row (max 68 bytes)

struct WriteParams {
  const void *src;
  int64_t n_rows;
  int64_t stride;
  const int64_t *row_ids;
  uint8_t *dst;
  int64_t dst_rows;
  int32_t *status;
  float c[16];
  float b[15];
  uint32_t wht_neg[4];
  const float *pi;  // dense: fp32 [128][128]
  const float *pit; // its transpose
  const float *S;   // prod3: fp32 [128][128]
  const float *St;  // its transpose
  const BucketTable *bt;  // nearest-centroid grid (n == 0: binary search over b)
};

// Stage the codebook grid in shared memory (16-byte pieces, all threads).
__device__ __forceinline__ void stage_grid(BucketTable *dst, const BucketTable *src) {
  constexpr int N16 = sizeof(BucketTable) / 16;
  for (int i = threadIdx.x; i < N16; i += blockDim.x)
    reinterpret_cast<uint4 *>(dst)[i] = reinterpret_cast<const uint4 *>(src)[i];
}

// Nearest-centroid index of y: the grid table when usable, else binary search.
template <int NB>
__device__ __forceinline__ uint32_t nearest(float y, const BucketTable &g, const float *sb);

template <int SRC>
__device__ __forceinline__ void load4(const void *src, int64_t row, int64_t stride, int lane,
                                      float (&x)[4]) {
  if (SRC == TQ_DTYPE_F32) {
    const float4 v = *reinterpret_cast<const float4 *>(static_cast<const float *>(src) +
                                                       row * stride + 4 * lane);
    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(src) +
                                                     row * stride + 4 * lane);
    x[0] = bf16_bits_to_f32(v.x & 0xFFFFu);
    x[1] = bf16_bits_to_f32(v.x >> 16);
    x[2] = bf16_bits_to_f32(v.y & 0xFFFFu);
    x[3] = bf16_bits_to_f32(v.y >> 16);
  }
}

// x / n rounded to nearest, given r = RN(1/n): q = RN(x r) is within one ulp of x / n,
// the residual x - q n is exact under a fused multiply-add, and one correction
// q + (x - q n) r rounded to nearest is RN(x / n) (Markstein's theorem for binary
// floating point with a correctly rounded reciprocal).  The theorem needs the
// residual and the quotient away from the subnormal range and 1/n normal; other
// operands (zeros included) take the IEEE division.
__device__ __forceinline__ float div_rn(float x, float n, float r) {
  const float q = __fmul_rn(x, r);
  if (fabsf(x) >= 0x1p-100f && fabsf(q) >= 0x1p-124f && n <= 0x1p125f)
    return __fmaf_rn(__fmaf_rn(-q, n, x), r, q);
  return __fdiv_rn(x, n);
}

// Canonical fp32 norm and u = x / n (u = 0 when n == 0).
__device__ __forceinline__ float norm_normalize(float (&x)[4]) {
  float p = __fadd_rn(__fadd_rn(__fmul_rn(x[0], x[0]), __fmul_rn(x[1], x[1])),
                      __fadd_rn(__fmul_rn(x[2], x[2]), __fmul_rn(x[3], x[3])));
#pragma unroll
  for (int h = 16; h >= 1; h >>= 1) p = __fadd_rn(p, __shfl_xor_sync(FULL_MASK, p, h));
  const float n = __fsqrt_rn(p);
  const float r = __frcp_rn(n);
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = (n == 0.0f) ? 0.0f : div_rn(x[e], n, r);
  return n;
}

// Number of boundaries strictly below y (binary search over NB sorted boundaries).
template <int NB>
__device__ __forceinline__ uint32_t bucket(float y, const float *sb) {
  uint32_t pos = 0;
#pragma unroll
  for (int step = (NB + 1) / 2; step >= 1; step >>= 1)
    if (y > sb[pos + step - 1]) pos += step;
  return pos;
}

template <int NB>
__device__ __forceinline__ uint32_t nearest(float y, const BucketTable &g, const float *sb) {
  return g.n ? bucket_grid(y, g.scale, g.offset, g.n, g.cnt, g.e) : bucket<NB>(y, sb);
}

// Pack one turbo4 / turbo3 row from per-lane indices (elements 4l..4l+3) and store
// it at dst + slot * row_bytes through the warp's staging buffer.
template <int FMT>
__device__ __forceinline__ void pack_store_turbo(const uint32_t (&idx)[4], float n, uint8_t *buf,
                                                 uint8_t *dst_row, int lane) {
  if (FMT == TQ_FMT_TURBO4) {
    if (lane == 0) *reinterpret_cast<float *>(buf) = n;
    buf[4 + 2 * lane] = (uint8_t)(idx[0] | (idx[1] << 4));
    buf[5 + 2 * lane] = (uint8_t)(idx[2] | (idx[3] << 4));
    __syncwarp();
    if (lane < 17)
      reinterpret_cast<uint32_t *>(dst_row)[lane] = reinterpret_cast<const uint32_t *>(buf)[lane];
  } else {  // turbo3: four 14-byte blocks {fp16 norm, qs[8], signs[4]}
    const int c = lane >> 3, q = lane & 7;
    uint8_t *blk = buf + 14 * c;
    if (q == 0) {
      const __half hn = __float2half_rn(n);
      const uint16_t bits = *reinterpret_cast<const uint16_t *>(&hn);
      blk[0] = (uint8_t)(bits & 0xFF);
      blk[1] = (uint8_t)(bits >> 8);
    }
    blk[2 + q] = (uint8_t)((idx[0] & 3) | ((idx[1] & 3) << 2) | ((idx[2] & 3) << 4) |
                           ((idx[3] & 3) << 6));
    const uint32_t nib = (idx[0] >> 2) | ((idx[1] >> 2) << 1) | ((idx[2] >> 2) << 2) |
                         ((idx[3] >> 2) << 3);
    const uint32_t other = __shfl_xor_sync(FULL_MASK, nib, 1);
    if ((q & 1) == 0) blk[10 + (q >> 1)] = (uint8_t)(nib | (other << 4));
    __syncwarp();
    if (lane < 14)
      reinterpret_cast<uint32_t *>(dst_row)[lane] = reinterpret_cast<const uint32_t *>(buf)[lane];
  }
  __syncwarp();
}

__device__ __forceinline__ bool slot_of(const WriteParams &p, int64_t row, int lane,
                                        int64_t *slot) {
  const int64_t s = p.row_ids ? p.row_ids[row] : row;
  if (s < 0 || s >= p.dst_rows) {
    if (lane == 0) atomicExch(p.status, (int32_t)DEVERR_ROW_OOB);
    return false;
  }
  *slot = s;
  return true;
}

// ------------------------------------------------------------------ WHT turbo4/turbo3
// Four threads per row (a warp takes eight rows).  Thread q holds the four 8-element
// chunks 32i + 8q .. 32i + 8q + 7 (i = 0..3) in registers, so one load instruction reads
// 64 contiguous bytes of each row, the butterfly stages 1, 2, 4, 32, 64 and the norm
// tree's strides 16, 8, 1 run inside the thread, and only butterfly stages 8, 16 and tree
// strides 4, 2 cross threads (shuffles within the row's four lanes).  The operation order
// is the canonical one -- four-element partial sums of squares combined over strides
// 16, 8, 4, 2, 1; butterfly stages of distance 1, 2, ..., 64 with the lower element taking
// a + b and the upper a - b -- so every value is bit-identical to a sequential fp32
// implementation of the same order.  Register element 8i + e is row element 32i + 8q + e.
constexpr int WT_THREADS = 256;
constexpr int WT_E = 32;     // elements per thread
constexpr int WT_REP = 16;   // copies of the grid table (one per half-warp lane)

// A thread's four chunks as loaded (bf16 bits or fp32), kept while the previous row is
// encoded.
template <int SRC>
struct Quarter {
  uint2 w[8];  // chunk i: w[2i], w[2i + 1] (eight bf16)
};
template <>
struct Quarter<TQ_DTYPE_F32> {
  float4 w[8];  // chunk i: w[2i], w[2i + 1]
};

// v16: bf16 rows are 16-byte aligned (one 16-byte load per chunk); fp32 rows always are.
template <int SRC>
__device__ __forceinline__ void load_quarter(const WriteParams &p, int64_t row, int q, bool v16,
                                             Quarter<SRC> &raw) {
  if constexpr (SRC == TQ_DTYPE_F32) {
    const float4 *s = reinterpret_cast<const float4 *>(static_cast<const float *>(p.src) + row * p.stride + 8 * q);
#pragma unroll
    for (int i = 0; i < 4; ++i) raw.w[2 * i] = s[8 * i], raw.w[2 * i + 1] = s[8 * i + 1];
  } else if (v16) {
    const uint4 *s = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.src) + row * p.stride + 8 * q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 c = s[4 * i];
      raw.w[2 * i] = make_uint2(c.x, c.y), raw.w[2 * i + 1] = make_uint2(c.z, c.w);
    }
  } else {
    const uint2 *s = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.src) + row * p.stride + 8 * q);
#pragma unroll
    for (int i = 0; i < 4; ++i) raw.w[2 * i] = s[8 * i], raw.w[2 * i + 1] = s[8 * i + 1];
  }
}

__device__ __forceinline__ void unpack_quarter(const Quarter<TQ_DTYPE_F32> &raw, float (&x)[WT_E]) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    x[4 * k] = raw.w[k].x, x[4 * k + 1] = raw.w[k].y, x[4 * k + 2] = raw.w[k].z, x[4 * k + 3] = raw.w[k].w;
}
__device__ __forceinline__ void unpack_quarter(const Quarter<TQ_DTYPE_BF16> &raw, float (&x)[WT_E]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    x[4 * k] = bf16_bits_to_f32(raw.w[k].x & 0xFFFFu), x[4 * k + 1] = bf16_bits_to_f32(raw.w[k].x >> 16);
    x[4 * k + 2] = bf16_bits_to_f32(raw.w[k].y & 0xFFFFu), x[4 * k + 3] = bf16_bits_to_f32(raw.w[k].y >> 16);
  }
}

// Canonical fp32 norm of the row (the four threads end with the same value), then u = x / n
// in place (u = 0 when n == 0).  Group g = 8i + 2q + h of the row is register group 2i + h.
__device__ __forceinline__ float quarter_norm_normalize(float (&x)[WT_E]) {
  float p[8];  // four-element partial sums of register groups 2i + h
#pragma unroll
  for (int k = 0; k < 8; ++k)
    p[k] = __fadd_rn(__fadd_rn(__fmul_rn(x[4 * k], x[4 * k]), __fmul_rn(x[4 * k + 1], x[4 * k + 1])),
                     __fadd_rn(__fmul_rn(x[4 * k + 2], x[4 * k + 2]), __fmul_rn(x[4 * k + 3], x[4 * k + 3])));
  float s[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    // stride 16 (chunk i + 2) and stride 8 (chunk i + 1), in this thread
    const float s16a = __fadd_rn(p[h], p[4 + h]), s16b = __fadd_rn(p[2 + h], p[6 + h]);
    s[h] = __fadd_rn(s16a, s16b);
  }
  // stride 4: threads q and q ^ 2; stride 2: q and q ^ 1; stride 1: h = 0 and 1 here
#pragma unroll
  for (int h = 0; h < 2; ++h) s[h] = __fadd_rn(s[h], __shfl_xor_sync(FULL_MASK, s[h], 2));
#pragma unroll
  for (int h = 0; h < 2; ++h) s[h] = __fadd_rn(s[h], __shfl_xor_sync(FULL_MASK, s[h], 1));
  const float n = __fsqrt_rn(__fadd_rn(s[0], s[1]));
  const float r = __frcp_rn(n);
  // Markstein's correction is exact when every nonzero |x| >= 2^-100 and n <= 2^24 (then
  // |q| >= 2^-124 and 1/n is normal); zeros come out as zeros.  Otherwise the guarded
  // per-element division.
  uint32_t mb = 0xFFFFFFFFu;  // min over elements of |x| bits - 1 (zero -> 0xFFFFFFFF)
#pragma unroll
  for (int j = 0; j < WT_E; ++j) mb = min(mb, (__float_as_uint(x[j]) & 0x7FFFFFFFu) - 1u);
  const bool fast = n <= 0x1p24f && mb >= 0x0D800000u - 1u;  // 0x0D800000: 2^-100
  if (n == 0.0f) {
#pragma unroll
    for (int j = 0; j < WT_E; ++j) x[j] = 0.0f;
  } else if (fast) {
#pragma unroll
    for (int j = 0; j < WT_E; ++j) {
      const float qq = __fmul_rn(x[j], r);
      x[j] = __fmaf_rn(__fmaf_rn(-qq, n, x[j]), r, qq);
    }
  } else {
#pragma unroll
    for (int j = 0; j < WT_E; ++j) x[j] = div_rn(x[j], n, r);
  }
  return n;
}

// Randomized Hadamard of the row: sign flips (bit j % 32 of word j / 32 for row element j;
// nq[i] = sign word i shifted down by 8q), the butterfly, times RN(1/sqrt(128)).
__device__ __forceinline__ void wht_quarter(float (&v)[WT_E], const uint32_t (&nq)[4], int q) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e)
      v[8 * i + e] = __uint_as_float(__float_as_uint(v[8 * i + e]) ^ ((nq[i] << (31 - e)) & 0x80000000u));
  auto stage = [&](int h, int hr) {  // row distance h = register distance hr, in this thread
#pragma unroll
    for (int k = 0; k < WT_E; ++k)
      if (!(k & hr)) {
        const float a = v[k], b = v[k + hr];
        v[k] = __fadd_rn(a, b);
        v[k + hr] = __fsub_rn(a, b);
      }
    (void)h;
  };
  stage(1, 1);
  stage(2, 2);
  stage(4, 4);
  // distances 8 and 16: partner thread q ^ 1, then q ^ 2; the lower one keeps v + o, the
  // upper one o - v, both as one fused o + (+-1) v (the product by +-1 is exact)
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    const float sgn = (q & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int k = 0; k < WT_E; ++k) {
      const float o = __shfl_xor_sync(FULL_MASK, v[k], m);
      v[k] = __fmaf_rn(sgn, v[k], o);
    }
  }
  stage(32, 8);
  stage(64, 16);
  const float inv_sqrt_d = __int_as_float(0x3DB504F3);  // fp32 nearest 1/sqrt(128)
#pragma unroll
  for (int k = 0; k < WT_E; ++k) v[k] = __fmul_rn(v[k], inv_sqrt_d);
}

// #{k : y > b_k}: the grid (copy l16 of cell t: boundary .x, count .y as integer bits) or,
// without GRID, binary search over the NB boundaries.
template <bool GRID, int NB>
__device__ __forceinline__ uint32_t cell_index(float y, const float2 *ce, int l16, float gs, float go, int gn,
                                               const float *sb) {
  if (GRID) {
    // unsigned round-down conversion: negative, -inf and NaN give 0, +inf saturates
    const uint32_t t = min(__float2uint_rd(fmaf(y, gs, go)), (uint32_t)(gn - 1));
    const float2 c = ce[t * WT_REP + l16];
    return __float_as_uint(c.y) + (y > c.x ? 1u : 0u);
  }
  return bucket<NB>(y, sb);
}

// Nearest-centroid indices of this thread's elements, packed into its part of the row
// record at row (4-byte aligned).  turbo4 (fp32 norm + 64 nibble bytes): chunk i fills
// word 1 + 4i + q; thread 0 writes the norm.  turbo3 (four 14-byte blocks {fp16 norm,
// qs[8] with the low two index bits of block element j at bits 2 (j % 4) of qs[j / 4],
// signs[4] with the high bit at bit j % 8 of signs[j / 8]}): chunk i is elements
// 8q .. 8q+7 of block i, i.e. qs[2q], qs[2q + 1] and signs[q].
template <int FMT, bool GRID>
__device__ __forceinline__ void pack_quarter(const float (&y)[WT_E], float n, const float2 *ce, int l16,
                                             float gs, float go, int gn, const float *sb, uint8_t *row,
                                             int q) {
  constexpr int NB = (FMT == TQ_FMT_TURBO4) ? 15 : 7;
  if (FMT == TQ_FMT_TURBO4) {
    uint32_t *w = reinterpret_cast<uint32_t *>(row);
    if (q == 0) w[0] = __float_as_uint(n);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) word |= cell_index<GRID, NB>(y[8 * i + e], ce, l16, gs, go, gn, sb) << (4 * e);
      w[1 + 4 * i + q] = word;
    }
  } else {
    const __half hn = __float2half_rn(n);
    const uint16_t nb = *reinterpret_cast<const uint16_t *>(&hn);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t idx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) idx[e] = cell_index<GRID, NB>(y[8 * i + e], ce, l16, gs, go, gn, sb);
      uint32_t lo = 0, sg = 0;  // qs[2q] | qs[2q + 1] << 8, signs[q]
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        lo |= (idx[e] & 3u) << (2 * e);
        sg |= (idx[e] >> 2) << e;
      }
      uint8_t *blk = row + 14 * i;  // 2-byte aligned
      if (q == 0) *reinterpret_cast<uint16_t *>(blk) = nb;
      *reinterpret_cast<uint16_t *>(blk + 2 + 2 * q) = (uint16_t)lo;
      blk[10 + q] = (uint8_t)sg;
    }
  }
}

// The WHT write's shared tables: the boundaries, the grid table (cell t, copy c at
// t * WT_REP + c: boundary .x, count .y as integer bits) and its scale, offset and size.
struct WhtTables {
  float sb[16];
  float2 ce[GRID_CELLS * WT_REP];
  float2 cell0[GRID_CELLS];  // one copy, read from memory
  float gs, go;
  int gn;
};

// Filled by every thread of the CTA (the caller synchronises again before use).
template <int FMT>
__device__ __forceinline__ void wht_tables_fill(const WriteParams &p, WhtTables &tb) {
  constexpr int NB = (FMT == TQ_FMT_TURBO4) ? 15 : 7;
  if (threadIdx.x < NB) tb.sb[threadIdx.x] = p.b[threadIdx.x];
  // each cell read from memory once (one latency for the whole table), then copied with
  // consecutive threads on consecutive entries
  for (int t = threadIdx.x; t < GRID_CELLS; t += blockDim.x)
    tb.cell0[t] = make_float2(p.bt->e[t], __uint_as_float((uint32_t)p.bt->cnt[t]));
  if (threadIdx.x == 0) tb.gs = p.bt->scale, tb.go = p.bt->offset, tb.gn = p.bt->n;
  __syncthreads();
  for (int k = threadIdx.x; k < GRID_CELLS * WT_REP; k += blockDim.x) tb.ce[k] = tb.cell0[k / WT_REP];
}

// Rows in groups of eight per warp (four threads per row): this warp takes row groups it,
// it + step, ...  The four threads of a row stay together (whole warps iterate while any
// row is left); the next group's source chunks and slot are loaded before this one is
// encoded.
template <int FMT, int SRC>
__device__ __forceinline__ void wht_rows(const WriteParams &p, const WhtTables &tb, int64_t it, int64_t step) {
  constexpr int RB = (FMT == TQ_FMT_TURBO4) ? 68 : 56;
  const float gs = tb.gs, go = tb.go;
  const int gn = tb.gn;
  const int q = threadIdx.x & 3, l16 = threadIdx.x & 15;
  uint32_t nq[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) nq[i] = p.wht_neg[i] >> (8 * q);
  const bool v16 = ((uintptr_t)p.src & 15) == 0 && ((p.stride * 2) & 15) == 0;
  const int64_t n_iter = (p.n_rows + 7) / 8;
  const int sub = (threadIdx.x & 31) >> 2;
  Quarter<SRC> raw;
  int64_t slot_next = -1;
  auto fetch = [&](int64_t i) {
    const int64_t row = i * 8 + sub;
    if (i < n_iter && row < p.n_rows) {
      load_quarter<SRC>(p, row, q, v16, raw);
      slot_next = p.row_ids ? p.row_ids[row] : row;
    }
  };
  fetch(it);
  for (; it < n_iter; it += step) {
    const int64_t row = it * 8 + sub;
    const bool live = row < p.n_rows;
    const int64_t slot = slot_next;
    const bool ok = live && slot >= 0 && slot < p.dst_rows;
    if (live && !ok && q == 0) atomicExch(p.status, (int32_t)DEVERR_ROW_OOB);
    float v[WT_E];
    if (ok) {
      unpack_quarter(raw, v);
    } else {
#pragma unroll
      for (int i = 0; i < WT_E; ++i) v[i] = 0.0f;
    }
    fetch(it + step);
    const float n = quarter_norm_normalize(v);  // shuffles: every lane of the warp takes part
    wht_quarter(v, nq, q);
    if (ok) {
      uint8_t *dst = p.dst + slot * RB;
      if (gn)
        pack_quarter<FMT, true>(v, n, tb.ce, l16, gs, go, gn, tb.sb, dst, q);
      else
        pack_quarter<FMT, false>(v, n, tb.ce, l16, gs, go, gn, tb.sb, dst, q);
    }
  }
}

template <int FMT, int SRC>
__global__ void __launch_bounds__(WT_THREADS) k_write_wht(const WriteParams p) {
  __shared__ WhtTables tb;
  pdl_trigger();
  wht_tables_fill<FMT>(p, tb);
  __syncthreads();
  pdl_wait();
  wht_rows<FMT, SRC>(p, tb, (int64_t)blockIdx.x * (WT_THREADS / 32) + (threadIdx.x >> 5),
                     (int64_t)gridDim.x * (WT_THREADS / 32));
}

// ------------------------------------------------- dense rotation (CUDA-core matvec)
// The matrices are staged once per CTA in shared memory, unpadded and in the
// orientation that makes lane l's accesses for outputs l + 32 m consecutive:
// R^T for y = R u, R for x_tilde = R^T y_hat, S^T for z = S r.  Staging issues all
// 16-byte loads before the first store, so it costs one memory latency.
__device__ __forceinline__ void stage128(float *dst, const float *src) {
  const float4 *s4 = reinterpret_cast<const float4 *>(src);
  float4 *d4 = reinterpret_cast<float4 *>(dst);
  constexpr int PER = D * D / 4 / (WARPS * 32);
  float4 v[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) v[i] = s4[threadIdx.x + i * WARPS * 32];
#pragma unroll
  for (int i = 0; i < PER; ++i) d4[threadIdx.x + i * WARPS * 32] = v[i];
}

template <int FMT, int SRC>
__global__ void __launch_bounds__(WARPS * 32) k_write_dense(const WriteParams p) {
  extern __shared__ __align__(16) float dsm[];
  constexpr int NMAT = (FMT == TQ_FMT_PROD3) ? 3 : 1;
  float *RT = dsm;                                                   // [128][128] R^T
  float *Rm = dsm + D * D;                                           // prod3: R
  float *ST = dsm + 2 * D * D;                                       // prod3: S^T
  float *vec = dsm + NMAT * D * D;                                   // [WARPS][3][128]
  uint8_t *ib = reinterpret_cast<uint8_t *>(vec + WARPS * 3 * D);    // [WARPS][128] indices
  uint8_t *rowbuf = ib + WARPS * D;                                  // [WARPS][ROWBUF]
  float *sb = reinterpret_cast<float *>(rowbuf + WARPS * ROWBUF);    // [16]
  __shared__ BucketTable grid;
  pdl_trigger();
  stage_grid(&grid, p.bt);
  stage128(RT, p.pit);
  if (FMT == TQ_FMT_PROD3) {
    stage128(Rm, p.pi);
    stage128(ST, p.St);
  }
  if (threadIdx.x < 15) sb[threadIdx.x] = p.b[threadIdx.x];
  __syncthreads();
  pdl_wait();
  constexpr int NB = (FMT == TQ_FMT_TURBO4) ? 15 : (FMT == TQ_FMT_TURBO3 ? 7 : 3);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *u = vec + warp * 3 * D;
  float *yh = u + D;
  float *rr = yh + D;
  uint8_t *myib = ib + warp * D;
  uint8_t *buf = rowbuf + warp * ROWBUF;
  for (int64_t row = (int64_t)blockIdx.x * WARPS + warp; row < p.n_rows;
       row += (int64_t)gridDim.x * WARPS) {
    int64_t slot;
    if (!slot_of(p, row, lane, &slot)) continue;
    float x[4];
    load4<SRC>(p.src, row, p.stride, lane, x);
    const float n = norm_normalize(x);
    *reinterpret_cast<float4 *>(u + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
    __syncwarp();
    float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int k = 0; k < D; ++k) {
      const float uk = u[k];
      const float *rt = RT + k * D + lane;  // (R u)_j = sum_k R^T[k][j] u_k
#pragma unroll
      for (int m = 0; m < 4; ++m) y[m] = fmaf(rt[32 * m], uk, y[m]);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) myib[lane + 32 * m] = (uint8_t)nearest<NB>(y[m], grid, sb);
    __syncwarp();
    uint32_t idx[4];
    const uint32_t w4 = *reinterpret_cast<const uint32_t *>(myib + 4 * lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) idx[e] = (w4 >> (8 * e)) & 0xFF;
    if (FMT != TQ_FMT_PROD3) {
      pack_store_turbo<FMT>(idx, n, buf, p.dst + slot * (FMT == TQ_FMT_TURBO4 ? 68 : 56), lane);
      continue;
    }
    // prod3: residual in the unrotated normalised space, its norm, and QJL signs.
#pragma unroll
    for (int m = 0; m < 4; ++m) yh[lane + 32 * m] = p.c[myib[lane + 32 * m]];
    __syncwarp();
    float r[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int k = 0; k < D; ++k) {
      const float yk = yh[k];
      const float *rk = Rm + k * D + lane;  // (R^T y)_j = sum_k R[k][j] y_k
#pragma unroll
      for (int m = 0; m < 4; ++m) r[m] = fmaf(rk[32 * m], yk, r[m]);
    }
    float g2 = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      r[m] = u[lane + 32 * m] - r[m];
      rr[lane + 32 * m] = r[m];
      g2 = fmaf(r[m], r[m], g2);
    }
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1) g2 += __shfl_xor_sync(FULL_MASK, g2, h);
    __syncwarp();
    float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int k = 0; k < D; ++k) {
      const float rk = rr[k];
      const float *st = ST + k * D + lane;  // (S r)_i = sum_k S^T[k][i] r_k
#pragma unroll
      for (int m = 0; m < 4; ++m) z[m] = fmaf(st[32 * m], rk, z[m]);
    }
    uint32_t sbits[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) sbits[m] = __ballot_sync(FULL_MASK, z[m] >= 0.0f);
    if (lane == 0) {
      reinterpret_cast<float *>(buf)[0] = n;
      reinterpret_cast<float *>(buf)[1] = sqrtf(g2);
#pragma unroll
      for (int m = 0; m < 4; ++m) reinterpret_cast<uint32_t *>(buf)[10 + m] = sbits[m];
    }
    buf[8 + lane] = (uint8_t)((idx[0] & 3) | ((idx[1] & 3) << 2) | ((idx[2] & 3) << 4) |
                              ((idx[3] & 3) << 6));
    __syncwarp();
    if (lane < 14)
      reinterpret_cast<uint32_t *>(p.dst + slot * 56)[lane] =
          reinterpret_cast<const uint32_t *>(buf)[lane];
    __syncwarp();
  }
}

// ---------------------------------------- dense rotation, small batches (one CTA per row)
// For the few rows of a decode step: thread j < 128 computes output coordinate j from row
// j of R read straight from L2 (no 64 KB staging) into registers before the wait on the
// previous kernel (R belongs to the immutable context), so after that wait the launch
// costs about one memory latency.  Norm, normalisation and packing follow the same
// canonical order as above.  Threads j >= 128 of a larger CTA only join the barriers.
struct RowScratch {
  float u[D];
  float grp[32];
  float sb[16];
  float nsh;
  BucketTable grid;
  alignas(16) uint8_t ib[D];
  alignas(16) uint8_t buf[ROWBUF];
};

// Before the wait: the boundaries, the grid table, R staged (padded rows) at Rs.
template <int NB>
__device__ __forceinline__ void dense_row_prologue(const WriteParams &p, RowScratch &sc, int j, float *Rs) {
  if (j == 0) {
#pragma unroll
    for (int k = 0; k < NB; ++k) sc.sb[k] = p.b[k];
  }
  stage_grid(&sc.grid, p.bt);
  stage_rows_padded(Rs, p.pi);
}

// After the wait, the first part of a row's encoding (the whole CTA takes the same row):
// its slot (-1 when out of range: flagged, nothing to write), the canonical norm n and
// u = x / n in sc.u (thread j < 128 holds element j; every thread takes the barriers).
template <int SRC>
__device__ __forceinline__ int64_t dense_row_normalize(const WriteParams &p, int64_t row, RowScratch &sc, int j,
                                                       float *n_out) {
  const int lane = j & 31;
  const bool act = j < D;
  // the source element is read before the slot is checked, so the two loads overlap
  float x = 0.f;
  if (act) {
    if (SRC == TQ_DTYPE_F32)
      x = static_cast<const float *>(p.src)[row * p.stride + j];
    else
      x = bf16_bits_to_f32(static_cast<const uint16_t *>(p.src)[row * p.stride + j]);
  }
  const int64_t slot = p.row_ids ? p.row_ids[row] : row;
  if (slot < 0 || slot >= p.dst_rows) {  // the same for every thread of the CTA
    if (j == 0) atomicExch(p.status, (int32_t)DEVERR_ROW_OOB);
    return -1;
  }
  if (act) {
    // canonical norm: groups of four (pairs summed first), then the butterfly over groups
    const float sq = __fmul_rn(x, x);
    const float a = __fadd_rn(sq, __shfl_xor_sync(FULL_MASK, sq, 1));
    const float g = __fadd_rn(a, __shfl_xor_sync(FULL_MASK, a, 2));
    if ((j & 3) == 0) sc.grp[j >> 2] = g;
  }
  __syncthreads();
  if (j < 32) {
    float pl = sc.grp[lane];
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1) pl = __fadd_rn(pl, __shfl_xor_sync(FULL_MASK, pl, h));
    if (lane == 0) sc.nsh = __fsqrt_rn(pl);
  }
  __syncthreads();
  const float n = sc.nsh;
  if (act) sc.u[j] = (n == 0.0f) ? 0.0f : __fdiv_rn(x, n);
  __syncthreads();
  *n_out = n;
  return slot;
}

// y_j = (R u)_j from row j of R (rrow: its padded row in shared memory), in k order.
__device__ __forceinline__ float row_times_u(const float *rrow, const float *u) {
  float y = 0.f;
#pragma unroll 8
  for (int k4 = 0; k4 < D / 4; ++k4) {
    const float4 r = *reinterpret_cast<const float4 *>(rrow + 4 * k4);
    y = fmaf(r.x, u[4 * k4], y);
    y = fmaf(r.y, u[4 * k4 + 1], y);
    y = fmaf(r.z, u[4 * k4 + 2], y);
    y = fmaf(r.w, u[4 * k4 + 3], y);
  }
  return y;
}

// After the wait: encode source row `row` into its slot (the whole CTA takes the same row).
template <int FMT, int SRC>
__device__ __forceinline__ void dense_row_body(const WriteParams &p, int64_t row, RowScratch &sc, int j,
                                               const float *Rs) {
  constexpr int NB = (FMT == TQ_FMT_TURBO4) ? 15 : 7;
  const int lane = j & 31;
  const bool act = j < D;
  float n;
  const int64_t slot = dense_row_normalize<SRC>(p, row, sc, j, &n);
  if (slot < 0) return;
  if (act) {
    const float y = row_times_u(Rs + j * RPAD, sc.u);
    sc.ib[j] = (uint8_t)nearest<NB>(y, sc.grid, sc.sb);
  }
  __syncthreads();
  if (j < 32) {
    const uint32_t w4 = *reinterpret_cast<const uint32_t *>(sc.ib + 4 * lane);
    const uint32_t idx[4] = {w4 & 0xFF, (w4 >> 8) & 0xFF, (w4 >> 16) & 0xFF, w4 >> 24};
    pack_store_turbo<FMT>(idx, n, sc.buf, p.dst + slot * (FMT == TQ_FMT_TURBO4 ? 68 : 56), lane);
  }
}

constexpr size_t ROW_SMEM = (size_t)D * RPAD * sizeof(float);  // R with padded rows

template <int FMT, int SRC>
__global__ void __launch_bounds__(D) k_write_dense_row(const WriteParams p) {
  extern __shared__ __align__(16) float rsm[];
  __shared__ RowScratch sc;
  dense_row_prologue<(FMT == TQ_FMT_TURBO4) ? 15 : 7>(p, sc, threadIdx.x, rsm);
  pdl_trigger();
  pdl_wait();
  dense_row_body<FMT, SRC>(p, blockIdx.x, sc, threadIdx.x, rsm);
}

// A prod3 row by one CTA (the decode step's few new keys): the same steps as the warp-per-row
// kernel above with thread j < 128 on coordinate j.  y = R u (row j of the staged R),
// x_tilde = R^T y_hat (column j of R) and z = S r (column j of S^T), R with padded rows and
// S^T in shared memory: no bank conflicts.
struct Prod3Scratch {
  RowScratch base;
  float yh[D];  // centroids of the indices
  float r[D];   // residual u - R^T y_hat
};

template <int SRC>
__device__ __forceinline__ void prod3_row_body(const WriteParams &p, int64_t row, Prod3Scratch &sc, const float *Rs,
                                               const float *STs, int j) {
  const int lane = j & 31, warp = j >> 5;
  const bool act = j < D;
  float n;
  const int64_t slot = dense_row_normalize<SRC>(p, row, sc.base, j, &n);
  if (slot < 0) return;
  if (act) {
    const uint32_t idx = nearest<3>(row_times_u(Rs + j * RPAD, sc.base.u), sc.base.grid, sc.base.sb);
    sc.base.ib[j] = (uint8_t)idx;
    sc.yh[j] = p.c[idx];
  }
  __syncthreads();
  if (act) {
    float xt = 0.f;  // (R^T y_hat)_j = sum_k R[k][j] y_hat_k
#pragma unroll 8
    for (int k = 0; k < D; ++k) xt = fmaf(Rs[k * RPAD + j], sc.yh[k], xt);
    sc.r[j] = sc.base.u[j] - xt;
  }
  __syncthreads();
  if (act) {
    float z = 0.f;  // (S r)_j = sum_k S^T[k][j] r_k
#pragma unroll 8
    for (int k = 0; k < D; ++k) z = fmaf(STs[k * D + j], sc.r[k], z);
    const uint32_t sbits = __ballot_sync(FULL_MASK, z >= 0.0f);  // elements 32 warp + lane
    uint8_t *buf = sc.base.buf;
    if (lane == 0) reinterpret_cast<uint32_t *>(buf)[10 + warp] = sbits;
    if (warp == 0) {  // gamma^2 in the warp kernel's order: lane l sums l + 32 m, then the lanes
      float g2 = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) g2 = fmaf(sc.r[lane + 32 * m], sc.r[lane + 32 * m], g2);
#pragma unroll
      for (int h = 16; h >= 1; h >>= 1) g2 += __shfl_xor_sync(FULL_MASK, g2, h);
      if (lane == 0) {
        reinterpret_cast<float *>(buf)[0] = n;
        reinterpret_cast<float *>(buf)[1] = sqrtf(g2);
      }
    }
    if (j < 32) {
      const uint32_t w4 = *reinterpret_cast<const uint32_t *>(sc.base.ib + 4 * j);
      buf[8 + j] = (uint8_t)((w4 & 3) | (((w4 >> 8) & 3) << 2) | (((w4 >> 16) & 3) << 4) | (((w4 >> 24) & 3) << 6));
    }
  }
  __syncthreads();
  if (j < 14) reinterpret_cast<uint32_t *>(p.dst + slot * 56)[j] = reinterpret_cast<const uint32_t *>(sc.base.buf)[j];
}

// ------------------------------------------------ decode step front (tq_decode_step)
// One launch for what a decode step does before its split-K kernel: the first q_ctas CTAs
// prepare q (tq_qprep.cuh; first, since theirs is the longest job), the next n encode the
// step's n new K rows, the last n its n new V rows (the small-batch dense write above).
// The three jobs are independent, so they share one wait on the previous kernel instead
// of three.
struct StepFrontParams {
  WriteParams wk, wv;
  QprepParams q;
  int n_rows;
  int q_ctas;
};

template <int KF, int VF, int SRC>
__global__ void __launch_bounds__(QWARPS * 32) k_step_front(const StepFrontParams sp) {
  extern __shared__ __align__(16) float fsm[];
  const int c = blockIdx.x - sp.q_ctas;  // row CTAs from 0
  if (c >= 0) {
    float *Rs = fsm;  // R with padded rows
    RowScratch &sc = *reinterpret_cast<RowScratch *>(fsm + D * RPAD);
    const bool v = c >= sp.n_rows;
    const int j = threadIdx.x;
    if (v)
      dense_row_prologue<(VF == TQ_FMT_TURBO4) ? 15 : 7>(sp.wv, sc, j, Rs);
    else
      dense_row_prologue<(KF == TQ_FMT_TURBO4) ? 15 : 7>(sp.wk, sc, j, Rs);
    pdl_trigger();
    pdl_wait();
    if (v)
      dense_row_body<VF, SRC>(sp.wv, c - sp.n_rows, sc, j, Rs);
    else
      dense_row_body<KF, SRC>(sp.wk, c, sc, j, Rs);
  } else {
    pdl_trigger();
    stage_rows_padded(fsm, sp.q.r);
    pdl_wait();
    prepare_q_body<false>(sp.q, blockIdx.x, sp.q_ctas, fsm);
  }
}

// The same front for randomized-WHT caches: the q CTAs as above (q_rot = R q with the
// stored WHT matrix), then ceil(n / 64) CTAs for the K rows and as many for the V rows,
// each warp encoding eight rows with the WHT write's four-threads-per-row body.
constexpr int FRONT_WHT_ROWS = WT_THREADS / 4;  // rows per row CTA
static_assert(QWARPS * 32 == WT_THREADS, "the front's CTAs are the WHT write's");

template <int KF, int VF, int SRC>
__global__ void __launch_bounds__(QWARPS * 32) k_step_front_wht(const StepFrontParams sp) {
  extern __shared__ __align__(16) float fsm[];
  const int c = blockIdx.x - sp.q_ctas;  // row CTAs from 0: K rows, then V rows
  if (c >= 0) {
    WhtTables &tb = *reinterpret_cast<WhtTables *>(fsm);
    const int rc = (sp.n_rows + FRONT_WHT_ROWS - 1) / FRONT_WHT_ROWS;  // row CTAs per tensor
    const bool v = c >= rc;
    const int cl = v ? c - rc : c;
    if (v)
      wht_tables_fill<VF>(sp.wv, tb);
    else
      wht_tables_fill<KF>(sp.wk, tb);
    __syncthreads();
    pdl_trigger();
    pdl_wait();
    const int64_t it = (int64_t)cl * QWARPS + (threadIdx.x >> 5), step = (int64_t)rc * QWARPS;
    if (v)
      wht_rows<VF, SRC>(sp.wv, tb, it, step);
    else
      wht_rows<KF, SRC>(sp.wk, tb, it, step);
  } else {
    pdl_trigger();
    stage_rows_padded(fsm, sp.q.r);
    pdl_wait();
    prepare_q_body<false>(sp.q, blockIdx.x, sp.q_ctas, fsm);
  }
}

// ------------------------------------------------------------------ V group quant
// One vgroup2 row by one warp: per 32-element group the fp16 min z and step s = (max - min) / 3,
// indices round((x - z) / s) clamped to 0..3 (48-byte record: 32 index bytes, then {s, z}
// per group).
template <int SRC>
__device__ __forceinline__ void vgroup_row(const WriteParams &p, int64_t row, int lane, uint8_t *buf) {
  int64_t slot;
  if (!slot_of(p, row, lane, &slot)) return;
  float x[4];
  load4<SRC>(p.src, row, p.stride, lane, x);
  float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
  for (int h = 1; h <= 4; h <<= 1) {  // lanes 8g..8g+7 hold group g
    mn = fminf(mn, __shfl_xor_sync(FULL_MASK, mn, h));
    mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, h));
  }
  mn = __fadd_rn(mn, 0.0f);
  mx = __fadd_rn(mx, 0.0f);
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
  const __half sh = __float2half_rn(s32);
  const __half zh = __float2half_rn(mn);
  const float s = __half2float(sh), z = __half2float(zh);
  uint32_t byte = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float c = 0.0f;
    if (s > 0.0f) c = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(x[e], z), s)), 0.0f), 3.0f);
    byte |= ((uint32_t)c) << (2 * e);
  }
  buf[lane] = (uint8_t)byte;
  if ((lane & 7) == 0) {
    const int g = lane >> 3;
    *reinterpret_cast<__half *>(buf + 32 + 4 * g) = sh;
    *reinterpret_cast<__half *>(buf + 34 + 4 * g) = zh;
  }
  __syncwarp();
  if (lane < 12)
    reinterpret_cast<uint32_t *>(p.dst + slot * 48)[lane] =
        reinterpret_cast<const uint32_t *>(buf)[lane];
  __syncwarp();
}

template <int SRC>
__global__ void __launch_bounds__(WARPS * 32) k_write_vgroup(const WriteParams p) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) uint8_t rowbuf[WARPS][ROWBUF];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t row = (int64_t)blockIdx.x * WARPS + warp; row < p.n_rows; row += (int64_t)gridDim.x * WARPS)
    vgroup_row<SRC>(p, row, lane, rowbuf[warp]);
}

// Decode step front for prod3 keys and vgroup2 values: the first q_ctas CTAs prepare q with
// its QJL sketch, the next n encode the n new K rows (one CTA per row, R and S^T staged
// before the wait), the last ceil(n / QWARPS) the V rows (one warp per row).
constexpr size_t FRONT_PV_SMEM = ((size_t)D * RPAD + D * D) * sizeof(float) + sizeof(Prod3Scratch);

template <int SRC>
__global__ void __launch_bounds__(QWARPS * 32) k_step_front_pv(const StepFrontParams sp) {
  extern __shared__ __align__(16) float fsm[];
  const int c = blockIdx.x - sp.q_ctas;  // row CTAs from 0: K rows, then V rows by warp
  if (c >= 0 && c < sp.n_rows) {
    float *Rs = fsm, *STs = fsm + D * RPAD;  // R with padded rows, S^T
    Prod3Scratch &sc = *reinterpret_cast<Prod3Scratch *>(fsm + D * RPAD + D * D);
    dense_row_prologue<3>(sp.wk, sc.base, threadIdx.x, Rs);
    stage_matrix(STs, sp.wk.St);
    pdl_trigger();
    pdl_wait();
    prod3_row_body<SRC>(sp.wk, c, sc, Rs, STs, threadIdx.x);
  } else if (c >= 0) {
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)(c - sp.n_rows) * QWARPS + warp;
    if (row < sp.n_rows) vgroup_row<SRC>(sp.wv, row, lane, reinterpret_cast<uint8_t *>(fsm) + warp * ROWBUF);
  } else {
    pdl_trigger();
    stage_rows_padded(fsm, sp.q.r);
    pdl_wait();
    prepare_q_body<true>(sp.q, blockIdx.x, sp.q_ctas, fsm);
  }
}

template <typename K>
cudaError_t launch_rows(K kernel, const WriteParams &p, int64_t n_rows, int num_sms, size_t smem,
                        int blocks_per_sm, cudaStream_t st) {
  if (smem > 48 * 1024) {
    cudaError_t e = kernel_smem_attr((const void *)kernel, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // One wave of resident CTAs (the kernels loop over rows): never more CTAs per SM than
  // fit at once, so no second, partial wave.
  int resident = 0;
  cudaError_t e = kernel_occupancy((const void *)kernel, WARPS * 32, smem, &resident);
  if (e != cudaSuccess) return e;
  if (resident >= 1 && resident < blocks_per_sm) blocks_per_sm = resident;
  int64_t want = (n_rows + WARPS - 1) / WARPS;
  int64_t cap = (int64_t)num_sms * blocks_per_sm;
  const int grid = (int)(want < cap ? want : cap);
  return launch_pdl(kernel, dim3(grid), dim3(WARPS * 32), smem, st, p);
}

// The WHT kernel (four threads per row): as many resident CTAs as the rows need.
template <typename K>
cudaError_t launch_thread_rows(K kernel, const WriteParams &p, int64_t n_rows, int num_sms, cudaStream_t st) {
  int resident = 0;
  cudaError_t e = kernel_occupancy((const void *)kernel, WT_THREADS, 0, &resident);
  if (e != cudaSuccess) return e;
  if (resident < 1) resident = 1;
  const int64_t want = (n_rows + WT_THREADS / 4 - 1) / (WT_THREADS / 4);  // four threads per row
  const int64_t cap = (int64_t)num_sms * resident;
  const int grid = (int)(want < cap ? want : cap);
  return launch_pdl(kernel, dim3(grid), dim3(WT_THREADS), 0, st, p);
}

WriteParams write_params(const tq_ctx *ctx, const WriteLaunch &w) {
  WriteParams p{};
  p.src = w.src;
  p.n_rows = w.n_rows;
  p.stride = w.stride;
  p.row_ids = w.row_ids;
  p.dst = w.dst;
  p.dst_rows = w.dst_rows;
  p.status = ctx->d_status;
  for (int k = 0; k < ctx->cb.K; ++k) p.c[k] = ctx->cb.c[k];
  for (int k = 0; k + 1 < ctx->cb.K; ++k) p.b[k] = ctx->cb.b[k];
  for (int i = 0; i < 4; ++i) p.wht_neg[i] = ctx->wht_neg[i];
  p.pi = ctx->d_pi;
  p.pit = ctx->d_pit;
  p.S = ctx->d_S;
  p.St = ctx->d_St;
  p.bt = ctx->d_bt;
  return p;
}

}  // namespace

cudaError_t launch_write(const tq_ctx *ctx, const WriteLaunch &w, cudaStream_t st) {
  const WriteParams p = write_params(ctx, w);
  const bool bf16 = (w.src_dtype == TQ_DTYPE_BF16);
  const int fmt = ctx->fmt;
  const int sms = ctx->num_sms;
  if (fmt == TQ_FMT_VGROUP2)
    return bf16 ? launch_rows(k_write_vgroup<TQ_DTYPE_BF16>, p, w.n_rows, sms, 0, 8, st)
                : launch_rows(k_write_vgroup<TQ_DTYPE_F32>, p, w.n_rows, sms, 0, 8, st);
  if (ctx->p.rotation == TQ_ROT_WHT && fmt != TQ_FMT_PROD3) {
    if (fmt == TQ_FMT_TURBO4)
      return bf16 ? launch_thread_rows(k_write_wht<TQ_FMT_TURBO4, TQ_DTYPE_BF16>, p, w.n_rows, sms, st)
                  : launch_thread_rows(k_write_wht<TQ_FMT_TURBO4, TQ_DTYPE_F32>, p, w.n_rows, sms, st);
    return bf16 ? launch_thread_rows(k_write_wht<TQ_FMT_TURBO3, TQ_DTYPE_BF16>, p, w.n_rows, sms, st)
                : launch_thread_rows(k_write_wht<TQ_FMT_TURBO3, TQ_DTYPE_F32>, p, w.n_rows, sms, st);
  }
  // Dense rotation on the tensor cores for 16-byte aligned bf16 rows (turbo4 / turbo3).
  if (write_tc_eligible(ctx, w)) return launch_write_tc(ctx, w, st);
  // A few rows (a decode step's new tokens): one CTA per row, R read from L2.
  if (w.n_rows <= SMALL_ROWS && fmt != TQ_FMT_PROD3) {
    const dim3 grid((unsigned)w.n_rows), block(D);
    auto kern = fmt == TQ_FMT_TURBO4
                    ? (bf16 ? k_write_dense_row<TQ_FMT_TURBO4, TQ_DTYPE_BF16> : k_write_dense_row<TQ_FMT_TURBO4, TQ_DTYPE_F32>)
                    : (bf16 ? k_write_dense_row<TQ_FMT_TURBO3, TQ_DTYPE_BF16> : k_write_dense_row<TQ_FMT_TURBO3, TQ_DTYPE_F32>);
    cudaError_t e = kernel_smem_attr((const void *)kern, (int)ROW_SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, block, ROW_SMEM, st, p);
  }
  // Dense rotation on the CUDA cores (prod3 always takes this path; its WHT variant
  // multiplies by the materialised WHT matrix, which the context stores as well).
  const size_t mats = (fmt == TQ_FMT_PROD3 ? 3 : 1) * (size_t)D * D * sizeof(float);
  const size_t smem = mats + WARPS * 3 * D * sizeof(float) + WARPS * D + WARPS * ROWBUF +
                      16 * sizeof(float);
  const int per_sm = fmt == TQ_FMT_PROD3 ? 1 : 2;
  switch (fmt) {
    case TQ_FMT_TURBO4:
      return bf16 ? launch_rows(k_write_dense<TQ_FMT_TURBO4, TQ_DTYPE_BF16>, p, w.n_rows, sms, smem, per_sm, st)
                  : launch_rows(k_write_dense<TQ_FMT_TURBO4, TQ_DTYPE_F32>, p, w.n_rows, sms, smem, per_sm, st);
    case TQ_FMT_TURBO3:
      return bf16 ? launch_rows(k_write_dense<TQ_FMT_TURBO3, TQ_DTYPE_BF16>, p, w.n_rows, sms, smem, per_sm, st)
                  : launch_rows(k_write_dense<TQ_FMT_TURBO3, TQ_DTYPE_F32>, p, w.n_rows, sms, smem, per_sm, st);
    default:
      return bf16 ? launch_rows(k_write_dense<TQ_FMT_PROD3, TQ_DTYPE_BF16>, p, w.n_rows, sms, smem, per_sm, st)
                  : launch_rows(k_write_dense<TQ_FMT_PROD3, TQ_DTYPE_F32>, p, w.n_rows, sms, smem, per_sm, st);
  }
}


bool step_front_eligible(const tq_ctx *k, const tq_ctx *v, const WriteLaunch &wk, const WriteLaunch &wv) {
  // dense: the small-batch dense write; WHT: the WHT write's row body.  Both contexts in
  // the same rotation family.
  auto ok = [](const tq_ctx *c, const WriteLaunch &w) {
    return (c->fmt == TQ_FMT_TURBO4 || c->fmt == TQ_FMT_TURBO3) && w.n_rows >= 1 && w.n_rows <= SMALL_ROWS &&
           (c->p.rotation == TQ_ROT_WHT || !write_tc_eligible(c, w));
  };
  return ok(k, wk) && ok(v, wv) && k->p.rotation == v->p.rotation && wk.n_rows == wv.n_rows &&
         wk.src_dtype == wv.src_dtype;
}

bool step_front_pv_eligible(const tq_ctx *k, const tq_ctx *v, const WriteLaunch &wk, const WriteLaunch &wv) {
  return k->fmt == TQ_FMT_PROD3 && v->fmt == TQ_FMT_VGROUP2 && wk.n_rows >= 1 && wk.n_rows <= SMALL_ROWS &&
         wk.n_rows == wv.n_rows && wk.src_dtype == wv.src_dtype;
}

cudaError_t launch_step_front_pv(const tq_ctx *k, const tq_ctx *v, const WriteLaunch &wk, const WriteLaunch &wv,
                                 const QprepParams &q, cudaStream_t st) {
  StepFrontParams sp{};
  sp.wk = write_params(k, wk);
  sp.wv = write_params(v, wv);
  sp.q = q;
  sp.n_rows = (int)wk.n_rows;
  sp.q_ctas = (q.n_q + QWARPS - 1) / QWARPS;
  static_assert(FRONT_PV_SMEM >= QPREP_SMEM && FRONT_PV_SMEM >= QWARPS * ROWBUF, "one dynamic area for every role");
  auto kern = wk.src_dtype == TQ_DTYPE_BF16 ? k_step_front_pv<TQ_DTYPE_BF16> : k_step_front_pv<TQ_DTYPE_F32>;
  cudaError_t e = kernel_smem_attr((const void *)kern, (int)FRONT_PV_SMEM);
  if (e != cudaSuccess) return e;
  const int grid = sp.n_rows + (sp.n_rows + QWARPS - 1) / QWARPS + sp.q_ctas;
  return launch_pdl(kern, dim3(grid), dim3(QWARPS * 32), FRONT_PV_SMEM, st, sp);
}

cudaError_t launch_step_front(const tq_ctx *k, const tq_ctx *v, const WriteLaunch &wk, const WriteLaunch &wv,
                              const QprepParams &q, cudaStream_t st) {
  StepFrontParams sp{};
  sp.wk = write_params(k, wk);
  sp.wv = write_params(v, wv);
  sp.q = q;
  sp.n_rows = (int)wk.n_rows;
  sp.q_ctas = (q.n_q + QWARPS - 1) / QWARPS;
  const bool bf16 = wk.src_dtype == TQ_DTYPE_BF16;
  const bool k4 = k->fmt == TQ_FMT_TURBO4, v4 = v->fmt == TQ_FMT_TURBO4;
  static_assert(ROW_SMEM + sizeof(RowScratch) <= QPREP_SMEM, "one dynamic shared area for both roles");
  auto pick = [&]() {
    if (bf16) {
      if (k4) return v4 ? k_step_front<TQ_FMT_TURBO4, TQ_FMT_TURBO4, TQ_DTYPE_BF16>
                        : k_step_front<TQ_FMT_TURBO4, TQ_FMT_TURBO3, TQ_DTYPE_BF16>;
      return v4 ? k_step_front<TQ_FMT_TURBO3, TQ_FMT_TURBO4, TQ_DTYPE_BF16>
                : k_step_front<TQ_FMT_TURBO3, TQ_FMT_TURBO3, TQ_DTYPE_BF16>;
    }
    if (k4) return v4 ? k_step_front<TQ_FMT_TURBO4, TQ_FMT_TURBO4, TQ_DTYPE_F32>
                      : k_step_front<TQ_FMT_TURBO4, TQ_FMT_TURBO3, TQ_DTYPE_F32>;
    return v4 ? k_step_front<TQ_FMT_TURBO3, TQ_FMT_TURBO4, TQ_DTYPE_F32>
              : k_step_front<TQ_FMT_TURBO3, TQ_FMT_TURBO3, TQ_DTYPE_F32>;
  };
  if (k->p.rotation == TQ_ROT_WHT) {
    static_assert(sizeof(WhtTables) <= QPREP_SMEM, "one dynamic shared area for both roles");
    auto pick_wht = [&]() {
      if (bf16) {
        if (k4) return v4 ? k_step_front_wht<TQ_FMT_TURBO4, TQ_FMT_TURBO4, TQ_DTYPE_BF16>
                          : k_step_front_wht<TQ_FMT_TURBO4, TQ_FMT_TURBO3, TQ_DTYPE_BF16>;
        return v4 ? k_step_front_wht<TQ_FMT_TURBO3, TQ_FMT_TURBO4, TQ_DTYPE_BF16>
                  : k_step_front_wht<TQ_FMT_TURBO3, TQ_FMT_TURBO3, TQ_DTYPE_BF16>;
      }
      if (k4) return v4 ? k_step_front_wht<TQ_FMT_TURBO4, TQ_FMT_TURBO4, TQ_DTYPE_F32>
                        : k_step_front_wht<TQ_FMT_TURBO4, TQ_FMT_TURBO3, TQ_DTYPE_F32>;
      return v4 ? k_step_front_wht<TQ_FMT_TURBO3, TQ_FMT_TURBO4, TQ_DTYPE_F32>
                : k_step_front_wht<TQ_FMT_TURBO3, TQ_FMT_TURBO3, TQ_DTYPE_F32>;
    };
    auto kern = pick_wht();
    cudaError_t e = kernel_smem_attr((const void *)kern, (int)QPREP_SMEM);
    if (e != cudaSuccess) return e;
    const int rc = (sp.n_rows + FRONT_WHT_ROWS - 1) / FRONT_WHT_ROWS;
    return launch_pdl(kern, dim3(2 * rc + sp.q_ctas), dim3(QWARPS * 32), QPREP_SMEM, st, sp);
  }
  auto kern = pick();
  cudaError_t e = kernel_smem_attr((const void *)kern, (int)QPREP_SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(2 * sp.n_rows + sp.q_ctas), dim3(QWARPS * 32), QPREP_SMEM, st, sp);
}

}  // namespace tq
