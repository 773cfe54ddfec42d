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
// preparation) and held in tensor memory for the item; K_hat and V_hat^T are decoded
// from the packed nibbles into 128-byte swizzled fp16 operand tiles in shared memory
// (byte permutes over the codebook's fp16 magnitudes, alpha-scaled); the softmax runs on
// the accumulator lanes (one row per thread pair, 64 columns each) in the log2 domain
// with the value norm folded into the exponent and a lazily raised running max (the O
// accumulator is rescaled in tensor memory only when the max grows by more than 2^8);
// P goes back into tensor memory as fp16 hi + lo over its own S columns, and the PV
// product takes it from there.  The products therefore read only K_hat and V_hat^T from
// shared memory.  All operand pairs are exact fp16 products accumulated in fp32, so the
// only rounding beyond fp32 is the fp16 centroid table, as in the decode.
//
// Per key tile the score products of the next tile run under this tile's softmax (two
// score accumulators in tensor memory), and the decode of the next key tile and of this
// value tile run under the products in flight; one warp issues the products and copies.
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

constexpr int PF_COMPUTE = 256;  // eight compute warps: warp w owns accumulator lanes 32 (w % 4)
                                 // .. + 31 (rows) and columns 64 (w / 4) .. + 63 of each accumulator
constexpr int PF_THREADS = PF_COMPUTE + 32;  // + one warp that issues the products and copies
constexpr int PF_KEYS = 128;     // keys per tile
static_assert(PF_KEYS == PF_TILE, "tile size shared with the host");
constexpr int T4_ROW = 68;
constexpr uint32_t RAW_BYTES = PF_KEYS * T4_ROW + 32;  // a packed tile + alignment slack
// Tensor memory (512 columns x 128 lanes, lane = row of the tile):
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0;    // S of even / odd key tiles: columns 0-127 / 128-255, fp32;
                                 // each tile's P (fp16 hi + lo) overwrites its own S
constexpr uint32_t COL_O = 256;  // O accumulator, fp32
constexpr uint32_t COL_Q = 384;  // Q_hi (columns 384-447) and Q_lo (448-511), fp16 pairs

constexpr uint32_t OFF_K = 0;                            // K_hat tile (swizzled fp16)
constexpr uint32_t OFF_VT = OFF_K + SW_TILE_BYTES;       // V_hat^T tile (swizzled fp16)
constexpr uint32_t OFF_RAWK = OFF_VT + SW_TILE_BYTES;    // packed K tile
constexpr uint32_t OFF_RAWV = OFF_RAWK + RAW_BYTES;      // packed V tiles of even / odd key tiles
constexpr uint32_t OFF_MISC = OFF_RAWV + 2 * RAW_BYTES;
static_assert(RAW_BYTES % 16 == 0, "bulk copies land 16-byte aligned");

struct PfMisc {
  uint64_t rawk_full;       // the packed K tile landed
  uint64_t rawv_full[2];    // the packed V tile of an even / odd key tile landed
  uint64_t s_done;          // the score products of a tile finished
  uint64_t pv_done;         // the PV products of a tile finished
  uint64_t k_ready;         // K_hat of the next tile stored (256 compute threads)
  uint64_t p_ready;         // P (tensor memory) and V_hat^T of a tile stored (256 compute threads)
  uint64_t drain;           // teardown after a failed wait: every issued product finished
  uint32_t tmem_addr;
  int abort_flag;
  alignas(16) float knorm[2][PF_KEYS];  // key norms of even / odd tiles (read as float4)
  alignas(16) float vnu[2][PF_KEYS];    // log2 of the value norms, clamped at -64 (float4)
  alignas(16) float nvs[2][PF_KEYS];    // 2^(vnu + P_SHIFT): the value norm as a
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
  int tiles_per_unit, sched_g, sched_v, vx, total_tiles, n_part;  // vx = 0: equal tile ranges
  uint32_t sched_q, sched_r;  // V / G and V % G (set_schedule)
  float sched_ginv, sched_inv;  // 1 / G and G / V
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

// Barrier over the 256 compute threads (barrier 1) that also ORs a failure flag across
// them, so all compute threads take the same branch afterwards.
__device__ __forceinline__ bool compute_sync_or(bool fail) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)fail)
      : "memory");
  return r != 0;
}

// S(j) = Q K_hat(j)^T over the 128 dims: Q_hi and Q_lo from tensor memory, K_hat from
// shared memory; 16 MMAs of K = 16 issued by one thread.
__device__ __forceinline__ void issue_scores(uint32_t tmem_s, uint32_t tmem_q, uint32_t sk) {
#pragma unroll
  for (int part = 0; part < 2; ++part) {
#pragma unroll
    for (int s = 0; s < 8; ++s)
      umma_ts<IDESC_F16>(tmem_s, tmem_q + 64 * part + 8 * s, sw128_desc(sk + sw128_kstep(s)), (part || s) ? 1u : 0u);
  }
}

// O (+)= P(j) V_hat(j) over the 128 keys: P from tensor memory, where it overwrote the
// tile's S -- keys 32 m .. 32 m + 31 sit at columns 32 m .. 32 m + 31 of the S block, 16
// columns of fp16 pairs hi then 16 lo -- and V_hat^T from shared memory.
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t svt, bool accumulate) {
#pragma unroll
  for (int part = 0; part < 2; ++part) {
#pragma unroll
    for (int s = 0; s < 8; ++s)
      umma_ts<IDESC_F16>(tmem_o, tmem_p + 32 * (s >> 1) + 16 * part + 8 * (s & 1), sw128_desc(svt + sw128_kstep(s)),
                         (accumulate || part || s) ? 1u : 0u);
  }
}

// Warps 0-7 compute (operand decode, softmax, probabilities); warp 8 issues the tensor-core
// products and the bulk copies, so the compute warps never wait for the tensor core's
// instruction queue.  The two sides meet only at mbarriers:
//   compute -> issuer: k_ready (K_hat of the next tile stored), p_ready (P of this tile in
//                      tensor memory and V_hat^T in shared memory);
//   issuer -> compute: s_done, pv_done (products finished), rawk_full / rawv_full
//                      (packed tiles landed).
// Per tile j the compute warps: wait S(j) | decode K_hat(j+1), signal | value norms(j) |
// read S(j), row max | exponentials, P(j) into S(j)'s columns | wait PV(j-1), rescale O,
// decode V_hat^T(j), signal.  The issuer: wait K_hat(j+1) and PV(j-1) (S(j+1) takes
// over P(j-1)'s columns), issue S(j+1) | wait P(j), issue PV(j).  Q and P reach the tensor core from tensor memory, so the products read
// only K_hat and V_hat^T from shared memory.  Every wait is bounded; a wait that gives up
// raises a CTA flag that makes later waits fail at once, and the compute warps leave
// together at their next group barrier.
__global__ void __launch_bounds__(PF_THREADS, 1) k_prefill_t4(const PrefillParams p) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t *smem = smem_dyn + ((1024u - (smem_addr(smem_dyn) & 1023u)) & 1023u);
  PfMisc &ms = *reinterpret_cast<PfMisc *>(smem + OFF_MISC);
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool issuer_warp = warp == PF_COMPUTE / 32;
  const bool issuer = tid == PF_COMPUTE;
  const int half = (warp >> 2) & 1;             // compute warps: column half 64 * half .. + 63
  const int r = (warp & 3) * 32 + (tid & 31);   // compute warps: tensor-memory lane = row
  pdl_trigger();

  if (warp == 0) tmem_alloc(smem_addr(&ms.tmem_addr), TMEM_COLS);
  if (tid == 0) {
    mbar_init(&ms.rawk_full, 1);
    mbar_init(&ms.rawv_full[0], 1);
    mbar_init(&ms.rawv_full[1], 1);
    mbar_init(&ms.s_done, 1);
    mbar_init(&ms.pv_done, 1);
    mbar_init(&ms.k_ready, PF_COMPUTE);
    mbar_init(&ms.p_ready, PF_COMPUTE);
    mbar_init(&ms.drain, 1);
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
  const uint32_t tS = tmem + lane_off + COL_S + 64 * half, tO = tmem + lane_off + COL_O + 64 * half;
  const uint32_t sk = smem_addr(smem + OFF_K), svt = smem_addr(smem + OFF_VT);
  const uint32_t klo[2] = {p.klo[0], p.klo[1]}, khi[2] = {p.khi[0], p.khi[1]};
  const uint32_t vlo[2] = {p.vlo[0], p.vlo[1]}, vhi[2] = {p.vhi[0], p.vhi[1]};
  // mbarrier parities, tracked by the threads that wait on each barrier (rawv: one bit per
  // buffer)
  uint32_t ph_rawk = 0, ph_rawv = 0, ph_s = 0, ph_pv = 0, ph_k = 0, ph_p = 0;
  // the issuer's counts of copies per barrier and of PV products (the n-th completes the
  // barrier's phase n), and whether it issued products (teardown after a failed wait)
  uint32_t n_rawk = 0, n_rawv0 = 0, n_rawv1 = 0, n_pv = 0;
  bool mma_issued = false;

  // Bounded wait for the phase of the given parity; fails at once when another thread has
  // given up already.
  auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
    if (*reinterpret_cast<volatile int *>(&ms.abort_flag)) return false;
    const bool done = mbar_wait_bounded(bar, parity, WAIT_LIMIT_NS);
    if (!done) atomicExch(&ms.abort_flag, 1);
    return done;
  };

  int t = cta_first_tile(p, (int)blockIdx.x);
  Item it;
  while (next_item(p, (int)blockIdx.x, t, it)) {
    __syncthreads();  // the previous item is finished by every warp
    if (*reinterpret_cast<volatile int *>(&ms.abort_flag)) break;
    const int qt = it.unit % p.n_qt, bk = it.unit / p.n_qt;
    const int b = bk / p.Hkv, kvh = bk % p.Hkv;
    const int start = min(max(p.q_start[b], 0), p.L - p.T);
    const int i0 = qt * p.qpt;
    const int nq = min(p.qpt, p.T - i0);
    const int rows = nq * p.gq;
    const int horizon = start + i0 + nq;  // keys [0, horizon) are visible to some row
    const int t0 = it.t0;
    const int j_end = min(it.t1, (horizon + PF_KEYS - 1) / PF_KEYS);
    const size_t unit_row0 = (size_t)bk * p.L;

    // Shared-memory address of the packed K (v = false) or V (v = true) rows of key tile j.
    auto raw_base = [&](int j, bool v) -> uint8_t * {
      return smem + (v ? OFF_RAWV + (uint32_t)(j & 1) * RAW_BYTES : OFF_RAWK);
    };
    auto raw_rows = [&](int j, bool v) {
      return raw_base(j, v) + (((unit_row0 + (size_t)j * PF_KEYS) * T4_ROW) & 15);
    };
    // Bulk copy of those rows (the issuer).
    auto issue_raw = [&](int j, bool v) {
      const int kf = j * PF_KEYS, nk = min(PF_KEYS, p.L - kf);
      const size_t ks = (unit_row0 + kf) * T4_ROW;
      const size_t a0 = ks & ~(size_t)15;
      const uint32_t bytes = (uint32_t)(((ks + (size_t)nk * T4_ROW + 15) & ~(size_t)15) - a0);
      uint64_t *bar = v ? &ms.rawv_full[j & 1] : &ms.rawk_full;
      if (!v) ++n_rawk;
      else if (j & 1) ++n_rawv1;
      else ++n_rawv0;
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(raw_base(j, v), (v ? p.vc : p.kc) + a0, bytes, bar);
    };

    // ---- the item's q rows into tensor memory and per-row data (compute warps); the
    // first copies (issuer)
    if (!issuer_warp) {
      // thread (row r, half): Q_hi (half 0) or Q_lo (half 1) of row r, 64 columns of fp16 pairs
      uint4 qv[16];
      const bool live = r < rows;
      const int qi = i0 + r / p.gq, h = kvh * p.gq + r % p.gq;
      const uint4 *qw = reinterpret_cast<const uint4 *>(p.qhl + ((size_t)(b * p.T + qi) * p.Hq + h) * 256 + 64 * half);
#pragma unroll
      for (int c = 0; c < 16; ++c) qv[c] = live ? qw[c] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int c0 = 0; c0 < 2; ++c0) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = qv[8 * c0 + c];
          w[4 * c] = v.x, w[4 * c + 1] = v.y, w[4 * c + 2] = v.z, w[4 * c + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + COL_Q + 64 * half + 32 * c0, w);
      }
      if (half == 0) {
        ms.rowpos[r] = live ? start + qi : -1;
        ms.rowscale[r] = live ? p.qsc[2 * ((size_t)(b * p.T + qi) * p.Hq + h)] : 0.f;
      }
    } else if (issuer && t0 < j_end) {
      issue_raw(t0, false);
      issue_raw(t0, true);
      if (t0 + 1 < j_end) issue_raw(t0 + 1, true);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (issuer_warp) {
      // ============ the issuer: products and copies, in the order the compute warps need
      if (issuer && t0 < j_end) {
        bool ok = wait(&ms.k_ready, ph_k);  // K_hat(t0)
        ph_k ^= 1u;
        if (ok) {
          tc_fence_after();
          issue_scores(tmem + COL_S + 128 * (t0 & 1), tmem + COL_Q, sk);
          umma_commit(&ms.s_done);
          mma_issued = true;
          if (t0 + 1 < j_end) issue_raw(t0 + 1, false);
        }
        for (int j = t0; ok && j < j_end; ++j) {
          if (j + 1 < j_end) {  // K_hat(j+1) stored (so S(j) finished reading K_hat(j)): S(j+1)
            ok = wait(&ms.k_ready, ph_k);
            ph_k ^= 1u;
            // S(j+1) overwrites P(j-1); products on different accumulators may run out of
            // issue order, so PV(j-1) must have finished
            // (PV n completes the barrier's phase n, and PV(j-2) finished before P(j-1) was
            // stored, so the barrier is at most one phase behind)
            if (ok && j > t0) ok = wait(&ms.pv_done, (n_pv - 1) & 1u);
            if (!ok) break;
            tc_fence_after();
            issue_scores(tmem + COL_S + 128 * ((j + 1) & 1), tmem + COL_Q, sk);
            umma_commit(&ms.s_done);
            if (j + 2 < j_end) issue_raw(j + 2, false);
          }
          ok = wait(&ms.p_ready, ph_p);  // P(j) and V_hat^T(j) stored: PV(j)
          ph_p ^= 1u;
          if (!ok) break;
          tc_fence_after();
          issue_pv(tmem + COL_O, tmem + COL_S + 128 * (j & 1), svt, j > t0);
          umma_commit(&ms.pv_done);
          ++n_pv;
          if (j + 2 < j_end) issue_raw(j + 2, true);  // into the buffer tile j used
        }
      }
      continue;  // to the item barrier
    }

    // ============ compute warps
    // K_hat: thread (key k, half hf) decodes 64 dims into eight 16-byte chunks.
    auto decode_k = [&](int j) {
      const int k = tid & 127, hf = tid >> 7;
      const uint8_t *row = raw_rows(j, false) + k * T4_ROW;
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
      const uint8_t *ra = raw_rows(j, true) + (2 * kp) * T4_ROW, *rb = ra + T4_ROW;
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
    // this thread's shared- and tensor-memory writes -> the tensor core
    auto signal = [&](uint64_t *bar) {
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar);
    };

    const int pos = ms.rowpos[r];
    const float rsc = ms.rowscale[r];
    const uint64_t rsc2 = pk2(rsc, rsc);
    float M = -INFINITY, l = 0.f;
    bool fail = false;
    if (t0 < j_end) {
      const bool f = !wait(&ms.rawk_full, ph_rawk);
      ph_rawk ^= 1u;
      if (!f) decode_k(t0);
      signal(&ms.k_ready);
    }
    for (int j = t0; j < j_end; ++j) {
      const int kf = j * PF_KEYS;
      bool f = !wait(&ms.s_done, ph_s);  // S(j): the key tile is free again
      ph_s ^= 1u;
      if (j + 1 < j_end) {
        if (!f) f = !wait(&ms.rawk_full, ph_rawk);
        ph_rawk ^= 1u;
        if (!f) decode_k(j + 1);
        signal(&ms.k_ready);
      }
      if (!f) f = !wait(&ms.rawv_full[j & 1], (ph_rawv >> (j & 1)) & 1u);
      ph_rawv ^= 1u << (j & 1);
      if (!f && tid < PF_KEYS) {  // value norms of tile j: log2 (running max), 2^(log2 + P_SHIFT)
        const bool in = kf + tid < p.L;  // past the end: stale bytes, weight 0
        const float nv = *reinterpret_cast<const float *>(raw_rows(j, true) + tid * T4_ROW);
        const float nu = in ? fmaxf(log2_approx(nv), -64.f) : -64.f;
        ms.vnu[j & 1][tid] = nu;
        ms.nvs[j & 1][tid] = in ? exp2_approx(nu + P_SHIFT) : 0.f;
      }
      f = __any_sync(FULL_MASK, f);  // warp-uniform from here (tensor-memory loads)
      tc_fence_after();
      // S(j) is read twice from tensor memory (max pass, exponential pass) rather than
      // held in 64 registers across the group barrier
      const uint32_t tSj = tS + 128 * (j & 1);
      float sv[32];
      if (!f) tmem_ld32(tSj, sv);
      if ((fail = compute_sync_or(f))) break;  // the value norms are in place
      const float4 *kn4 = reinterpret_cast<const float4 *>(&ms.knorm[j & 1][64 * half]);
      const float4 *nu4 = reinterpret_cast<const float4 *>(&ms.vnu[j & 1][64 * half]);
      // every row of the tile sees every key of this tile unless it holds the diagonal
      const bool full = kf + PF_KEYS - 1 <= start + i0;
      // scaled score (log2 units) of columns c, c + 1 of this thread's half plus add, -inf
      // where masked
      auto scaled = [&](float s0, float s1, float k0, float k1, int c, uint64_t add) -> uint64_t {
        uint64_t v2 = fma2(mul2(pk2(s0, s1), pk2(k0, k1)), rsc2, add);
        if (!full) {
          float a, b2;
          upk2(v2, a, b2);
          const int kc = kf + 64 * half + c;
          v2 = pk2(kc <= pos ? a : -INFINITY, kc + 1 <= pos ? b2 : -INFINITY);
        }
        return v2;
      };
      float bm = -INFINITY;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        if (c0) tmem_ld32(tSj + c0, sv);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 kn = kn4[c0 / 4 + c4], nu = nu4[c0 / 4 + c4];
          float ua, ub;
          upk2(scaled(sv[4 * c4], sv[4 * c4 + 1], kn.x, kn.y, c0 + 4 * c4, pk2(nu.x, nu.y)), ua, ub);
          bm = fmaxf(bm, fmaxf(ua, ub));
          upk2(scaled(sv[4 * c4 + 2], sv[4 * c4 + 3], kn.z, kn.w, c0 + 4 * c4 + 2, pk2(nu.z, nu.w)), ua, ub);
          bm = fmaxf(bm, fmaxf(ua, ub));
        }
      }
      ms.pmax[half][r] = bm;
      if ((fail = compute_sync_or(false))) break;
      bm = fmaxf(ms.pmax[0][r], ms.pmax[1][r]);
      const bool raise = bm > M + RESCALE_SLACK;  // also taken while M is -inf; both halves agree
      const float alpha = raise ? exp2_approx(M - bm) : 1.f;
      if (raise) {
        M = bm;
        l *= alpha;
      }
      {
        // P(j) = 2^7 2^(s - M) n_v as fp16 hi + lo, written over S(j) chunk by chunk: the
        // 32 columns of a chunk are read before its 16 hi + 16 lo words replace them
        const float Mu = (M == -INFINITY) ? 0.f : M;
        const uint64_t nmu2 = pk2(-Mu, -Mu);
        const float4 *nv4 = reinterpret_cast<const float4 *>(&ms.nvs[j & 1][64 * half]);
        uint64_t l2 = pk2(0.f, 0.f);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          tmem_ld32(tSj + c0, sv);
          uint32_t pw[32];  // fp16 pairs: hi of columns c0 + 2i, + 1 in pw[i], lo in pw[16 + i]
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 kn = kn4[c0 / 4 + c4], nv = nv4[c0 / 4 + c4];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int c = 4 * c4 + 2 * h2;
              const uint64_t d2 = h2 ? scaled(sv[c], sv[c + 1], kn.z, kn.w, c0 + c, nmu2)
                                     : scaled(sv[c], sv[c + 1], kn.x, kn.y, c0 + c, nmu2);
              float da, db;
              upk2(d2, da, db);
              const uint64_t ex2 = pk2(exp2_approx(da), exp2_approx(db));  // 0 where masked
              l2 = add2(l2, ex2);
              const uint64_t pv2 = mul2(ex2, h2 ? pk2(nv.z, nv.w) : pk2(nv.x, nv.y));
              float pa, pb;
              upk2(pv2, pa, pb);
              const __half2 hi = __floats2half2_rn(pa, pb);
              const float2 hf = __half22float2(hi);
              float la, lb;
              upk2(sub2(pv2, pk2(hf.x, hf.y)), la, lb);
              const __half2 lo = __floats2half2_rn(la, lb);
              pw[2 * c4 + h2] = *reinterpret_cast<const uint32_t *>(&hi);
              pw[16 + 2 * c4 + h2] = *reinterpret_cast<const uint32_t *>(&lo);
            }
          }
          tmem_st32(tSj + c0, pw);
        }
        float la, lb;
        upk2(l2, la, lb);
        l += la + lb;
      }
      // PV(j-1) finished: O and the value tile are free
      f = false;
      if (j > t0) {
        f = !__all_sync(FULL_MASK, wait(&ms.pv_done, ph_pv));
        ph_pv ^= 1u;
        tc_fence_after();
        // tensor-memory loads and stores are warp-collective: the warp rescales its rows
        // together (factor 1 where the row's max stayed)
        if (!f && __any_sync(FULL_MASK, raise)) {
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            float o[32];
            tmem_ld32(tO + c0, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tO + c0, o);
          }
        }
      }
      if (!f) decode_v(j);
      signal(&ms.p_ready);  // also after a failed wait: the count stays whole
    }
    bool f = fail;
    if (!f && t0 < j_end) {  // the last PV of the item
      f = !__all_sync(FULL_MASK, wait(&ms.pv_done, ph_pv));
      ph_pv ^= 1u;
      tc_fence_after();
    }
    // ---- the item's partial for row r: (max, sum, O)
    ms.lsum[half][r] = l;
    if (!compute_sync_or(f)) {
      const bool row_live = r < rows;
      const int qi = i0 + r / p.gq, h = kvh * p.gq + r % p.gq;
      float *dst = p.part + ((size_t)((size_t)(b * p.T + qi) * p.Hq + h) * p.n_part + it.slot) * PARTIAL_FLOATS;
      const bool any = t0 < j_end;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        float o[32];
        if (any) {
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
  }

  if (issuer && *reinterpret_cast<volatile int *>(&ms.abort_flag)) {
    atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
    // let copies and products still in flight finish before the CTA leaves: copy n of a
    // barrier completes its phase n, so waiting for the last one's parity returns at once
    // when it has landed
    if (n_rawk) (void)mbar_wait_bounded(&ms.rawk_full, (n_rawk - 1) & 1u, WAIT_LIMIT_NS);
    if (n_rawv0) (void)mbar_wait_bounded(&ms.rawv_full[0], (n_rawv0 - 1) & 1u, WAIT_LIMIT_NS);
    if (n_rawv1) (void)mbar_wait_bounded(&ms.rawv_full[1], (n_rawv1 - 1) & 1u, WAIT_LIMIT_NS);
    if (mma_issued) {
      umma_commit(&ms.drain);
      (void)mbar_wait_bounded(&ms.drain, 0, WAIT_LIMIT_NS);
    }
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
  // the tiles split over one CTA per SM in proportion (ranges differ by at most one tile)
  s->grid = (int)(total < k->num_sms ? total : k->num_sms);
  const int shortest = (int)(total / s->grid);
  s->tiles_per_cta = (int)((total + s->grid - 1) / s->grid);
  s->n_part = (s->tiles_per_unit + shortest - 1) / shortest + 1;
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
  p.tiles_per_unit = s.tiles_per_unit, p.vx = 0;
  if (!set_schedule(p, s.grid, s.total_tiles)) return cudaErrorInvalidValue;
  p.total_tiles = s.total_tiles, p.n_part = s.n_part;
  p.qhl = ws.qhl, p.qsc = ws.qsc, p.part = ws.partials;
  for (int i = 0; i < 2; ++i) {
    p.klo[i] = k->f16.lo[i], p.khi[i] = k->f16.hi[i];
    p.vlo[i] = v->f16.lo[i], p.vhi[i] = v->f16.hi[i];
  }
  p.status = k->d_status;
  cudaError_t e = kernel_smem_attr((const void *)k_prefill_t4, (int)SMEM_PF);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_prefill_t4, dim3(s.grid), dim3(PF_THREADS), SMEM_PF, st, p);
}

}  // namespace tq
