// Chunked prefill attention over the compressed cache ("turboquant_plus: how the turbo4
// KV format came back", section 9 prefill table: prompt chunks attend to the turbo4
// cache, which by then already holds the chunk's own keys and values).  Query i of
// sequence b sits at position q_start[b] + i and attends to keys 0 .. q_start[b] + i.
//
// With many queries per KV head the scores and the PV product are dense contractions,
// so they run on the 5th-generation tensor cores: per work item (batch, KV head, tile
// of 128 rows = 128 / g queries x g q-heads) and per 128-key tile,
//   S[128 rows x 128 keys]  = (Q_hi + Q_lo) K_hat^T          tcgen05, fp32 in tensor memory
//   O[128 rows x 128 dims] += (P_hi + P_lo) V_hat              tcgen05, fp32 in tensor memory
// Q is rotated, scaled and split into fp16 hi + lo parts once (the decode's q
// preparation); K_hat and V_hat^T are decoded from the packed nibbles into 128-byte
// swizzled fp16 operand tiles in shared memory (byte permutes over the codebook's fp16
// magnitudes, alpha-scaled); the softmax runs on the accumulator lanes (one row per
// thread pair, 64 columns each) in the log2 domain with the value norm folded into the
// exponent and a lazily raised running max (the O accumulator is rescaled in tensor
// memory only when the max grows by more than 2^8); P goes back to shared memory as
// fp16 hi + lo.  All operand pairs are exact fp16 products accumulated in fp32, so the
// only rounding beyond fp32 is the fp16 centroid table, as in the decode.
//
// Per key tile the score products of the next tile run under this tile's softmax (two
// score accumulators in tensor memory), and the decode of the next key tile and of this
// value tile run under the products in flight.
//
// The (unit, key tile) sequence is split over one persistent CTA per SM in contiguous
// ranges (stream-K, as the decode), each (unit, CTA) pair writing a partial
// (max, sum, O) per row; the decode's combine merges them and un-rotates.
#include <math.h>
#include <stddef.h>

#include "tq_decode_common.cuh"
#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_tc.cuh"

namespace tq {

namespace {

constexpr int PF_THREADS = 256;  // eight warps: warp w owns accumulator lanes 32 (w % 4) .. + 31
                                 // (rows) and columns 64 (w / 4) .. + 63 of each accumulator
constexpr int PF_KEYS = 128;     // keys per tile
static_assert(PF_KEYS == PF_TILE, "tile size shared with the host");
constexpr int T4_ROW = 68;
constexpr uint32_t RAW_BYTES = PF_KEYS * T4_ROW + 32;  // a packed tile + alignment slack
constexpr uint32_t TMEM_COLS = 512;                    // S of even / odd tiles: columns 0-127 /
                                                       // 128-255, O: 256-383

constexpr uint32_t OFF_QH = 0;
constexpr uint32_t OFF_QL = OFF_QH + SW_TILE_BYTES;
constexpr uint32_t OFF_K = OFF_QL + SW_TILE_BYTES;
constexpr uint32_t OFF_VT = OFF_K + SW_TILE_BYTES;
constexpr uint32_t OFF_PH = OFF_VT + SW_TILE_BYTES;
constexpr uint32_t OFF_PL = OFF_PH + SW_TILE_BYTES;
constexpr uint32_t OFF_RAWK = OFF_PL + SW_TILE_BYTES;
constexpr uint32_t OFF_RAWV = OFF_RAWK + RAW_BYTES;
constexpr uint32_t OFF_MISC = OFF_RAWV + RAW_BYTES;
static_assert(RAW_BYTES % 16 == 0, "bulk copies land 16-byte aligned");

struct PfMisc {
  uint64_t rawk_full;       // the packed K tile landed
  uint64_t rawv_full;       // the packed V tile landed
  uint64_t s_done;          // the score products of a tile finished
  uint64_t pv_done;         // the PV products of a tile finished
  uint32_t tmem_addr;
  int abort_flag;
  alignas(16) float knorm[2][PF_KEYS];  // key norms of even / odd tiles (read as float4)
  alignas(16) float vnu[PF_KEYS];       // log2 of the value norms, clamped at -64 (float4)
  alignas(16) float nvs[PF_KEYS];       // 2^(vnu + P_SHIFT): the value norm as a
                                        // probability factor (float4)
  float rowscale[128];      // power-of-two scale of each row's q operand
  int rowpos[128];          // position of each row's query; -1 for padding rows
  float pmax[2][128];       // per-tile row maxima of the two column halves
  float lsum[2][128];       // row sums of the two column halves (end of an item)
};
static_assert(offsetof(PfMisc, knorm) % 16 == 0 && offsetof(PfMisc, vnu) % 16 == 0 &&
                  offsetof(PfMisc, nvs) % 16 == 0 && OFF_MISC % 16 == 0,
              "per-key arrays are read with 16-byte loads");
constexpr uint32_t SMEM_PF = OFF_MISC + sizeof(PfMisc) + 1024;  // + slack to align to 1024
static_assert(SMEM_PF <= 227 * 1024, "shared memory budget");

struct PrefillParams {
  const uint8_t *kc;
  const uint8_t *vc;
  const int32_t *q_start;   // [B] position of each sequence's first chunk query
  int B, T, Hq, Hkv, L, gq, qpt, n_qt;
  int tiles_per_unit, tiles_per_cta, total_tiles, n_part;
  const uint32_t *qhl;      // prepared q: [B*T*Hq][256 words], hi then lo fp16
  const float *qsc;         // [B*T*Hq][2] power-of-two scales
  float *part;              // [B*T*Hq][n_part][PARTIAL_FLOATS]
  uint32_t klo[2], khi[2], vlo[2], vhi[2];  // byte planes of the K / V fp16 magnitudes
  int32_t *status;
};

// Two-wide fp32 arithmetic (one instruction for two lanes of a register pair; each lane
// rounds exactly as the scalar operation).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// One thread issues the 16 products D (+)= A_hi B^T + A_lo B^T over K = 128.
__device__ __forceinline__ void issue_pair(uint32_t tmem_d, uint32_t a_hi, uint32_t a_lo, uint32_t b,
                                           bool accumulate) {
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    const uint32_t a = part ? a_lo : a_hi;
#pragma unroll
    for (int s = 0; s < 8; ++s)
      umma<IDESC_F16>(tmem_d, sw128_desc(a + sw128_kstep(s)), sw128_desc(b + sw128_kstep(s)),
                      (accumulate || part || s) ? 1u : 0u);
  }
}

__global__ void __launch_bounds__(PF_THREADS, 1) k_prefill_t4(const PrefillParams p) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t *smem = smem_dyn + ((1024u - (smem_addr(smem_dyn) & 1023u)) & 1023u);
  PfMisc &ms = *reinterpret_cast<PfMisc *>(smem + OFF_MISC);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int half = warp >> 2;              // column half: 64 * half .. + 63
  const int r = (warp & 3) * 32 + (tid & 31);  // accumulator lane = row of the tile
  pdl_trigger();

  if (warp == 0) tmem_alloc(smem_addr(&ms.tmem_addr), TMEM_COLS);
  if (tid == 0) {
    mbar_init(&ms.rawk_full, 1);
    mbar_init(&ms.rawv_full, 1);
    mbar_init(&ms.s_done, 1);
    mbar_init(&ms.pv_done, 1);
    ms.abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // q, the caches and the workspace may be written by the previous kernel
  if (tid == 0) {
    for (int b = 0; b < p.B; ++b)
      if (p.q_start[b] < 0 || p.q_start[b] > p.L - p.T) atomicExch(p.status, (int32_t)DEVERR_SEQLEN);
  }
  const uint32_t tmem = ms.tmem_addr;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + lane_off + 64 * half, tO = tmem + 256 + lane_off + 64 * half;
  const uint32_t sqh = smem_addr(smem + OFF_QH), sql = smem_addr(smem + OFF_QL);
  const uint32_t sk = smem_addr(smem + OFF_K), svt = smem_addr(smem + OFF_VT);
  const uint32_t sph = smem_addr(smem + OFF_PH), spl = smem_addr(smem + OFF_PL);
  const uint32_t klo[2] = {p.klo[0], p.klo[1]}, khi[2] = {p.khi[0], p.khi[1]};
  const uint32_t vlo[2] = {p.vlo[0], p.vlo[1]}, vhi[2] = {p.vhi[0], p.vhi[1]};
  uint32_t rawk_phase = 0, rawv_phase = 0, s_phase = 0, pv_phase = 0;
  bool rawk_pending = false, rawv_pending = false, s_pending = false, pv_pending = false;

  // Bounded wait on an mbarrier by every thread, then a CTA-wide verdict.
  auto wait_all = [&](uint64_t *bar, uint32_t &phase) -> bool {
    if (!mbar_wait_bounded(bar, phase, WAIT_LIMIT_NS)) atomicExch(&ms.abort_flag, 1);
    phase ^= 1u;
    tc_fence_after();
    __syncthreads();
    return *reinterpret_cast<volatile int *>(&ms.abort_flag) == 0;
  };

  int t = blockIdx.x * p.tiles_per_cta;
  Item it;
  bool ok = true;
  while (ok && next_item(p, (int)blockIdx.x, t, it)) {
    const int qt = it.unit % p.n_qt, bk = it.unit / p.n_qt;
    const int b = bk / p.Hkv, kvh = bk % p.Hkv;
    const int start = min(max(p.q_start[b], 0), p.L - p.T);
    const int i0 = qt * p.qpt;
    const int nq = min(p.qpt, p.T - i0);
    const int rows = nq * p.gq;
    const int horizon = start + i0 + nq;  // keys [0, horizon) are visible to some row
    const int j_end = min(it.t1, (horizon + PF_KEYS - 1) / PF_KEYS);
    const size_t unit_row0 = (size_t)bk * p.L;

    // ---- the item's q tile (hi, lo) and per-row data
    __syncthreads();  // the previous item's readers are done with the shared tiles
    for (int i = tid; i < 128 * 16; i += PF_THREADS) {
      const int row = i >> 4, ch = i & 15;  // chunk ch: dims 8 ch .. 8 ch + 7
      uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
      if (row < rows) {
        const int qi = i0 + row / p.gq, h = kvh * p.gq + row % p.gq;
        const uint4 *qw = reinterpret_cast<const uint4 *>(p.qhl + ((size_t)(b * p.T + qi) * p.Hq + h) * 256);
        hi = qw[ch];
        lo = qw[16 + ch];
      }
      *reinterpret_cast<uint4 *>(smem + OFF_QH + sw128_offset(row, 8 * ch)) = hi;
      *reinterpret_cast<uint4 *>(smem + OFF_QL + sw128_offset(row, 8 * ch)) = lo;
    }
    if (tid < 128) {
      const bool live = tid < rows;
      const int qi = i0 + tid / p.gq, h = kvh * p.gq + tid % p.gq;
      ms.rowpos[tid] = live ? start + qi : -1;
      ms.rowscale[tid] = live ? p.qsc[2 * ((size_t)(b * p.T + qi) * p.Hq + h)] : 0.f;
    }
    // Bulk copy of the packed K (v = false) or V (v = true) rows of key tile j.
    auto issue_raw = [&](int j, bool v) {
      const int kf = j * PF_KEYS, nk = min(PF_KEYS, p.L - kf);
      const size_t ks = (unit_row0 + kf) * T4_ROW;
      const size_t a0 = ks & ~(size_t)15;
      const uint32_t bytes = (uint32_t)(((ks + (size_t)nk * T4_ROW + 15) & ~(size_t)15) - a0);
      uint64_t *bar = v ? &ms.rawv_full : &ms.rawk_full;
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(smem + (v ? OFF_RAWV : OFF_RAWK), (v ? p.vc : p.kc) + a0, bytes, bar);
    };
    // Packed rows of tile j in a staging buffer (16-byte aligned copies).
    auto raw_rows = [&](int j, uint32_t off) {
      return smem + off + (((unit_row0 + (size_t)j * PF_KEYS) * T4_ROW) & 15);
    };
    // K_hat: thread (key k, half hf) decodes 64 dims into eight 16-byte chunks.
    auto decode_k = [&](int j) {
      const int k = tid & 127, hf = tid >> 7;
      const uint8_t *row = raw_rows(j, OFF_RAWK) + k * T4_ROW;
      uint32_t w[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) w[c] = *reinterpret_cast<const uint32_t *>(row + 4 + 32 * hf + 4 * c);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t d[4];
        decode8<0x5140u, 0x7362u>(w[c], klo, khi, d);
        *reinterpret_cast<uint4 *>(smem + OFF_K + sw128_offset(k, 64 * hf + 8 * c)) = make_uint4(d[0], d[1], d[2], d[3]);
      }
      // rows past the cache's end hold stale bytes: a zero norm keeps them finite
      if (hf == 0) ms.knorm[j & 1][k] = (j * PF_KEYS + k < p.L) ? *reinterpret_cast<const float *>(row) : 0.f;
    };
    // V_hat^T: thread (key pair kp, dim group dg) writes (key 2kp, key 2kp+1) pairs of 32
    // dims into rows d of the transposed tile.
    auto decode_v = [&](int j) {
      const int kp = tid & 63, dg = tid >> 6;
      const uint8_t *ra = raw_rows(j, OFF_RAWV) + (2 * kp) * T4_ROW, *rb = ra + T4_ROW;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t wa = *reinterpret_cast<const uint32_t *>(ra + 4 + 16 * dg + 4 * w);
        const uint32_t wb = *reinterpret_cast<const uint32_t *>(rb + 4 + 16 * dg + 4 * w);
        // byte i of zlo = (nibble of key a, nibble of key b) of dim 2i, of zhi: dim 2i + 1
        const uint32_t zlo = (wa & 0x0F0F0F0Fu) | ((wb << 4) & 0xF0F0F0F0u);
        const uint32_t zhi = ((wa >> 4) & 0x0F0F0F0Fu) | (wb & 0xF0F0F0F0u);
        uint32_t e[4], o[4];
        decode8<0x5140u, 0x7362u>(zlo, vlo, vhi, e);  // dims 0, 2, 4, 6 of this word
        decode8<0x5140u, 0x7362u>(zhi, vlo, vhi, o);  // dims 1, 3, 5, 7
        const int d0 = 32 * dg + 8 * w;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          *reinterpret_cast<uint32_t *>(smem + OFF_VT + sw128_offset(d0 + 2 * m, 2 * kp)) = e[m];
          *reinterpret_cast<uint32_t *>(smem + OFF_VT + sw128_offset(d0 + 2 * m + 1, 2 * kp)) = o[m];
        }
      }
    };
    auto cta_sync_for_mma = [&]() {  // generic smem writes -> tensor core, all threads
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    };

    if (tid == 0 && it.t0 < j_end) {
      issue_raw(it.t0, false);
      issue_raw(it.t0, true);
    }
    rawk_pending = rawv_pending = it.t0 < j_end;
    cta_sync_for_mma();
    const int pos = ms.rowpos[r];
    const float rsc = ms.rowscale[r];
    const uint64_t rsc2 = pk2(rsc, rsc);
    float M = -INFINITY, l = 0.f;
    bool o_init = false;
    if (it.t0 < j_end) {  // S(t0) in flight before the loop
      if ((ok = wait_all(&ms.rawk_full, rawk_phase))) {
        rawk_pending = false;
        decode_k(it.t0);
        cta_sync_for_mma();
        if (tid == 0) {
          issue_pair(tmem + 128 * (it.t0 & 1), sqh, sql, sk, false);
          umma_commit(&ms.s_done);
          if (it.t0 + 1 < j_end) issue_raw(it.t0 + 1, false);
        }
        s_pending = true;
        rawk_pending = it.t0 + 1 < j_end;
      }
    }

    // Per tile j (S(j) issued into accumulator j % 2; the packed K of tile j+1 and V of
    // tile j on their way; PV(j-1) issued):
    //   wait S(j) | decode K_hat(j+1), issue S(j+1) | softmax(j) into registers |
    //   wait PV(j-1) | rescale O, store P(j) | decode V_hat^T(j) | issue PV(j)
    // so the score products of the next tile run under this tile's softmax and the PV
    // products of the previous one.  All threads take every phase together: at this
    // size the phases are short and the tensor core's operand reads and the threads'
    // shared-memory traffic are kept apart.
    for (int j = it.t0; ok && j < j_end; ++j) {
      const int kf = j * PF_KEYS;
      if (!(ok = wait_all(&ms.s_done, s_phase))) break;
      s_pending = false;
      if (j + 1 < j_end) {  // the key tile is free: decode the next one, start its scores
        if (!(ok = wait_all(&ms.rawk_full, rawk_phase))) break;
        rawk_pending = false;
        decode_k(j + 1);
        cta_sync_for_mma();
        if (tid == 0) {
          issue_pair(tmem + 128 * ((j + 1) & 1), sqh, sql, sk, false);
          umma_commit(&ms.s_done);
          if (j + 2 < j_end) issue_raw(j + 2, false);
        }
        s_pending = true;
        rawk_pending = j + 2 < j_end;
      }
      if (!(ok = wait_all(&ms.rawv_full, rawv_phase))) break;
      rawv_pending = false;
      if (tid < PF_KEYS) {  // value norms of tile j: log2 (running max), 2^(log2 + P_SHIFT)
        const bool in = kf + tid < p.L;  // past the end: stale bytes, weight 0
        const float nv = *reinterpret_cast<const float *>(raw_rows(j, OFF_RAWV) + tid * T4_ROW);
        const float nu = in ? fmaxf(log2_approx(nv), -64.f) : -64.f;
        ms.vnu[tid] = nu;
        ms.nvs[tid] = in ? exp2_approx(nu + P_SHIFT) : 0.f;
      }

      // ---- online softmax over this thread's 64 columns of row r, into registers
      float sf[64];
      const uint32_t tSj = tS + 128 * (j & 1);
      tmem_ld32(tSj, *reinterpret_cast<float(*)[32]>(&sf[0]));
      tmem_ld32(tSj + 32, *reinterpret_cast<float(*)[32]>(&sf[32]));
      __syncthreads();  // the value norms are in place
      const float4 *kn4 = reinterpret_cast<const float4 *>(&ms.knorm[j & 1][64 * half]);
      const float4 *nu4 = reinterpret_cast<const float4 *>(&ms.vnu[64 * half]);
      // every row of the tile sees every key of this tile unless it holds the diagonal
      const bool full = kf + PF_KEYS - 1 <= start + i0;
      uint64_t sc2[32];  // scaled scores (log2 units) of column pairs, -inf where masked
      float bm = -INFINITY;
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 kn = kn4[c4], nu = nu4[c4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int c = 4 * c4 + 2 * h2;
          const uint64_t t2 = mul2(pk2(sf[c], sf[c + 1]), h2 ? pk2(kn.z, kn.w) : pk2(kn.x, kn.y));
          uint64_t u2 = fma2(t2, rsc2, h2 ? pk2(nu.z, nu.w) : pk2(nu.x, nu.y));
          uint64_t v2 = mul2(t2, rsc2);
          if (!full) {
            float a, b2, ua, ub;
            upk2(v2, a, b2);
            upk2(u2, ua, ub);
            const bool va = kf + 64 * half + c <= pos, vb = kf + 64 * half + c + 1 <= pos;
            v2 = pk2(va ? a : -INFINITY, vb ? b2 : -INFINITY);
            u2 = pk2(va ? ua : -INFINITY, vb ? ub : -INFINITY);
          }
          sc2[2 * c4 + h2] = v2;
          float ua, ub;
          upk2(u2, ua, ub);
          bm = fmaxf(bm, fmaxf(ua, ub));
        }
      }
      ms.pmax[half][r] = bm;
      __syncthreads();
      bm = fmaxf(ms.pmax[0][r], ms.pmax[1][r]);
      const bool raise = bm > M + RESCALE_SLACK;  // also taken while M is -inf; both halves agree
      const float alpha = raise ? exp2_approx(M - bm) : 1.f;
      if (raise) {
        M = bm;
        l *= alpha;
      }
      const float Mu = (M == -INFINITY) ? 0.f : M;
      const uint64_t mu2 = pk2(Mu, Mu);
      const float4 *nv4 = reinterpret_cast<const float4 *>(&ms.nvs[64 * half]);
      uint64_t l2 = pk2(0.f, 0.f);
      uint32_t ph[32], pl[32];  // P(j) of this thread's columns as fp16x2 hi and lo words
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 nv = nv4[c4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float da, db;
          upk2(sub2(sc2[2 * c4 + h2], mu2), da, db);
          const uint64_t ex2 = pk2(exp2_approx(da), exp2_approx(db));  // 0 where masked
          l2 = add2(l2, ex2);
          // 2^7 2^(s - M) n_v, split into fp16 hi + lo
          const uint64_t pv2 = mul2(ex2, h2 ? pk2(nv.z, nv.w) : pk2(nv.x, nv.y));
          float pa, pb;
          upk2(pv2, pa, pb);
          const __half2 hi = __floats2half2_rn(pa, pb);
          const float2 hf = __half22float2(hi);
          float la, lb;
          upk2(sub2(pv2, pk2(hf.x, hf.y)), la, lb);
          const __half2 lo = __floats2half2_rn(la, lb);
          ph[2 * c4 + h2] = *reinterpret_cast<const uint32_t *>(&hi);
          pl[2 * c4 + h2] = *reinterpret_cast<const uint32_t *>(&lo);
        }
      }
      {
        float la, lb;
        upk2(l2, la, lb);
        l += la + lb;
      }

      // ---- PV(j-1) finished: O, the probability tile and the value tile are free
      if (pv_pending) {
        if (!(ok = wait_all(&ms.pv_done, pv_phase))) break;
        pv_pending = false;
      }
      // tensor-memory loads and stores are warp-collective: the warp rescales its rows
      // together (factor 1 where the row's max stayed)
      if (o_init && __any_sync(FULL_MASK, raise)) {
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          float o[32];
          tmem_ld32(tO + c0, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tO + c0, o);
        }
      }
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        *reinterpret_cast<uint4 *>(smem + OFF_PH + sw128_offset(r, 64 * half + 8 * ch)) =
            make_uint4(ph[4 * ch], ph[4 * ch + 1], ph[4 * ch + 2], ph[4 * ch + 3]);
        *reinterpret_cast<uint4 *>(smem + OFF_PL + sw128_offset(r, 64 * half + 8 * ch)) =
            make_uint4(pl[4 * ch], pl[4 * ch + 1], pl[4 * ch + 2], pl[4 * ch + 3]);
      }
      decode_v(j);
      cta_sync_for_mma();
      if (tid == 0) {
        issue_pair(tmem + 256, sph, spl, svt, o_init);
        umma_commit(&ms.pv_done);
        if (j + 1 < j_end) issue_raw(j + 1, true);  // every thread is done with the packed V
      }
      pv_pending = true;
      rawv_pending = j + 1 < j_end;
      o_init = true;
    }
    if (ok && pv_pending) {
      ok = wait_all(&ms.pv_done, pv_phase);
      if (ok) pv_pending = false;
    }
    if (!ok) break;

    // ---- the item's partial for each live row: (max, sum, O)
    ms.lsum[half][r] = l;
    __syncthreads();
    const int row_live = r < rows;
    const int qi = i0 + r / p.gq, h = kvh * p.gq + r % p.gq;
    float *dst = p.part + ((size_t)((size_t)(b * p.T + qi) * p.Hq + h) * p.n_part + it.slot) * PARTIAL_FLOATS;
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
      float o[32];
      if (o_init) {
        tmem_ld32(tO + c0, o);  // warp-collective: every lane loads
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
      }
      if (row_live) {
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[6 + 64 * half + c0 + i] = (M == -INFINITY) ? 0.f : o[i];
      }
    }
    if (row_live && half == 0) {
      dst[0] = M;
      dst[1] = (M == -INFINITY) ? 0.f : ms.lsum[0][r] + ms.lsum[1][r];
      dst[2] = dst[3] = dst[4] = dst[5] = 0.f;
    }
  }

  if (!ok && tid == 0) {
    atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
    // let copies and products still in flight finish before the CTA leaves
    if (rawk_pending) (void)mbar_wait_bounded(&ms.rawk_full, rawk_phase, WAIT_LIMIT_NS);
    if (rawv_pending) (void)mbar_wait_bounded(&ms.rawv_full, rawv_phase, WAIT_LIMIT_NS);
    if (s_pending) (void)mbar_wait_bounded(&ms.s_done, s_phase, WAIT_LIMIT_NS);
    if (pv_pending) (void)mbar_wait_bounded(&ms.pv_done, pv_phase, WAIT_LIMIT_NS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool prefill_shape(const tq_ctx *k, int B, int T, int Hq, int Hkv, int L, PrefillShape *s) {
  s->B = B, s->T = T, s->Hq = Hq, s->Hkv = Hkv, s->L = L;
  s->gq = Hq / Hkv;
  if (s->gq < 1 || s->gq > 128 || 128 % s->gq != 0) return false;
  s->qpt = 128 / s->gq;
  s->n_qt = (T + s->qpt - 1) / s->qpt;
  const int64_t units = (int64_t)B * Hkv * s->n_qt;
  s->tiles_per_unit = (L + PF_TILE - 1) / PF_TILE;
  const int64_t total = units * s->tiles_per_unit;
  if (total > INT32_MAX || (int64_t)B * T * Hq > INT32_MAX / 256) return false;
  s->total_tiles = (int)total;
  const int64_t tpc = (total + k->num_sms - 1) / k->num_sms;
  s->tiles_per_cta = (int)(tpc < 1 ? 1 : tpc);
  s->grid = (int)((total + s->tiles_per_cta - 1) / s->tiles_per_cta);
  s->n_part = (s->tiles_per_unit + s->tiles_per_cta - 1) / s->tiles_per_cta + 1;
  // the q preparation and the workspace see the B*T queries of Hq heads as a batch
  DecodeShape &d = s->q;
  d = DecodeShape{};
  d.B = B * T, d.Hq = Hq, d.Hkv = Hkv, d.L = L, d.gq = s->gq;
  d.pv = false;
  d.n_part = s->n_part;
  return true;
}

cudaError_t launch_prefill(const tq_ctx *k, const tq_ctx *v, const uint8_t *kc, const uint8_t *vc,
                           const int32_t *q_start, const PrefillShape &s, const Workspace &ws,
                           cudaStream_t st) {
  PrefillParams p{};
  p.kc = kc, p.vc = vc, p.q_start = q_start;
  p.B = s.B, p.T = s.T, p.Hq = s.Hq, p.Hkv = s.Hkv, p.L = s.L, p.gq = s.gq, p.qpt = s.qpt, p.n_qt = s.n_qt;
  p.tiles_per_unit = s.tiles_per_unit, p.tiles_per_cta = s.tiles_per_cta;
  p.total_tiles = s.total_tiles, p.n_part = s.n_part;
  p.qhl = ws.qhl, p.qsc = ws.qsc, p.part = ws.partials;
  for (int i = 0; i < 2; ++i) {
    p.klo[i] = k->f16.lo[i], p.khi[i] = k->f16.hi[i];
    p.vlo[i] = v->f16.lo[i], p.vhi[i] = v->f16.hi[i];
  }
  p.status = k->d_status;
  cudaError_t e = cudaFuncSetAttribute(k_prefill_t4, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_PF);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_prefill_t4, dim3(s.grid), dim3(PF_THREADS), SMEM_PF, st, p);
}

}  // namespace tq
