// Fused decode attention over the packed cache ("TurboQuant fused Triton kernels
// deep dive", tricks 1-3): q is rotated once, every key is scored straight from
// its 4-bit indices, online softmax runs over key tiles split across the SMs,
// values are dequantized in registers, and the output is un-rotated once.
//
// Kernels (tq_decode_attention launches two, k_prepare_q and k_partial_t4 with the merge
// fused; the stage-by-stage calls, the store and larger unit counts use k_combine too):
//   k_prepare_q  q_rot = R q (one warp per query), pre-scaled by
//                log2(e) * scale / alpha and by a power of two, split into fp16
//                hi + lo parts (the tensor-core operand).
//   k_partial_t4 persistent: one CTA per SM takes a contiguous range of 240-key tiles
//                of the (batch, KV head, group of 4 or 8 q-heads) units laid end to
//                end, writing one partial (max, sum, acc) per unit it touches.  A
//                producer warp streams the K and V tiles into shared memory with 1-D
//                bulk async copies on a four-stage mbarrier ring; fifteen consumer
//                warps each take 16 keys of a tile, turn nibble pairs into fp16x2
//                centroid pairs (a conflict-free shared-memory table, or byte
//                permutes for a tunable share of the words), and run the score and
//                PV products as m16n8k16 MMAs with fp32 accumulators.
//                The CTA that completes a unit's partials merges them and writes its
//                outputs (the fused combine).
//   k_combine    log-sum-exp merge of the splits, 1/sum, un-rotation R^T o.
//
// MMA operand layout (one warp, 16 keys, 4 q-heads per column group):
//   score  S^T[16 keys x 8] = K_hat[16 keys x 128] Q^T : column 2h holds q_hi of
//          head h and column 2h+1 its q_lo, so the two add to the fp32-accurate score.
//   PV     O^T[128 x 8] += V_hat^T[128 x 16 keys] P^T : columns again hi/lo pairs.
//   Heads fill the N = 8 columns exactly for four q-heads per KV head, so no MMA
//   row is padding.  Probabilities move from the score accumulator layout to the
//   PV operand layout with four shuffles per 16 keys.
// Centroids enter as fp16 values alpha * c; alpha (chosen on the host) minimises
// the fp16 rounding error of the table and is divided out through q and in the
// combine.
#include <math.h>
#include <string.h>

#include <cstring>

#include "tq_decode_common.cuh"
#include "tq_qprep.cuh"
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int CWARPS = 15;            // consumer warps (16 keys each per tile)
constexpr int TILE = 16 * CWARPS;     // keys per pipeline stage (240)
static_assert(TILE == T4_TILE, "tile size shared with the host");
constexpr int NTHREADS = (CWARPS + 1) * 32;  // + one producer warp; one CTA per SM
constexpr int NSTAGE = 4;             // pipeline depth (about 128 KB in flight per SM)
constexpr int T4_ROW = 68;
constexpr int T3_ROW = 56;            // four 14-byte blocks of the 2+1 layout
constexpr int STAGE_BUF = 16352;      // >= 240 * 68 + 2 * 15, multiple of 32

// For 8 queries per CTA: q_rot = R q and, with SKETCH, the QJL sketch S q, each
// pre-scaled and split into the fp16 hi + lo tensor-core operands (tq_qprep.cuh).
template <bool SKETCH>
__global__ void __launch_bounds__(QWARPS * 32) k_prepare_q(const QprepParams p) {
  extern __shared__ __align__(16) float qsm[];
  pdl_trigger();
  stage_rows_padded(qsm, p.r);
  pdl_wait();
  prepare_q_body<SKETCH>(p, blockIdx.x, gridDim.x, qsm);
}

struct PartialParams {
  const uint8_t *kc;
  const uint8_t *vc;
  const int32_t *seq_lens;
  int B, Hq, Hkv, L, gq, n_hg;
  int tiles_per_unit, sched_g, sched_v, vx, total_tiles, n_part;
  uint32_t sched_q, sched_r;  // V / G and V % G (set_schedule)
  float sched_ginv, sched_inv;  // 1 / G and G / V
  const uint32_t *qhl;
  const float *qsc;
  float *part;
  float *scores;
  int withhold_first_tile;                  // failure test: the producer never copies tile 0
  uint32_t kc16[8], vc16[8];                // signed fp16 centroids (K, V), two per word
  uint32_t klo[2], khi[2], vlo[2], vhi[2];  // byte-permute tables (K and V codebooks)
  int32_t *status;
  // fused combine: out != null makes the CTA that completes a unit's partials merge them,
  // un-rotate (R row-major of the value rotation, or null) and write the unit's outputs
  float *out;
  const float *r;
  float inv_vscale;   // 1 / (2^P_SHIFT * alpha_V)
  int32_t *unit_done;  // [units] CTAs that have written their partial of the unit
};
constexpr int PREFETCH_TILES = 4;  // tiles per CTA pulled into L2 before the previous kernel ends
constexpr int FIN_MAX = 8;  // units one CTA may complete (the host fuses only below this)

// Shared memory of one CTA, as offsets from the start of dynamic shared memory.
// The 64 KB table lut[b][s] (slots s < 32: key table, s >= 32: value table; entry =
// (c[b & 15], c[b >> 4]) as fp16x2) sits at shared-window address 0x10000 when the
// device reserves the usual 1 KB at the window start, so a lookup's address
// (b << 8) | (4 * slot) is one byte permute of the packed word and the table base
// rides in the load's immediate.  Lane l reads slot l (keys) or 32 + l (values): a
// warp's 32 lookups hit 32 distinct banks.  With turbo3 keys the key slots of row b
// hold the spread sign bits of sign byte b instead.  Eight stage buffers (K and V of NSTAGE
// stages) and the merge scratch are packed around the table.
struct SmemHead {
  float osm[CWARPS][4][D];              // per-warp accumulators of 4 heads, for the merge
  uint64_t full[NSTAGE];
  uint64_t empty[NSTAGE];
  float mw[CWARPS][8];
  float lw[CWARPS][8];
  int abort_flag;
  int n_units;                          // fused combine: the units whose partials this CTA
  int units[FIN_MAX];                   // wrote; after the counts, the ones it completed
};
// The next work item's rotated q (fp16 hi and lo operand halves of up to 8 heads, 512 B
// each) and its per-head scales, copied in by the producer ahead of the consumers.
struct QStage {
  uint64_t full;    // producer: scales stored, then the q copies' bytes
  uint64_t empty;   // consumer warps: q taken into registers
  float qs[8];
  uint32_t pad[4];
  uint32_t q[8][128];
};
constexpr uint32_t STAGE_A_OFF = (sizeof(SmemHead) + 15) & ~15u;
constexpr uint32_t LUT_OFF = LUT_WINDOW - RESERVED_SMEM;
constexpr uint32_t STAGE_B_OFF = LUT_OFF + 256 * 64 * 4;
constexpr uint32_t QSTAGE_OFF = STAGE_B_OFF + 6 * STAGE_BUF;
constexpr uint32_t SMEM_BYTES = QSTAGE_OFF + sizeof(QStage);
static_assert(QSTAGE_OFF % 16 == 0 && offsetof(QStage, q) % 16 == 0, "bulk-copy destinations");
static_assert(SMEM_BYTES + RESERVED_SMEM <= 228 * 1024, "shared memory of one SM");
static_assert(STAGE_A_OFF + 2 * STAGE_BUF <= LUT_OFF, "two stage buffers below the table");
static_assert(NSTAGE == 4, "stage buffer placement assumes four stages");

// Stage buffer i (0..3: K of stage i, 4..7: V of stage i - 4).
__device__ __forceinline__ uint8_t *stage_buf(uint8_t *smem, int i) {
  return smem + (i < 2 ? STAGE_A_OFF + i * STAGE_BUF : STAGE_B_OFF + (i - 2) * STAGE_BUF);
}

// Table lookup of byte I of w.  FIXED: the table is at window address LUT_WINDOW and
// the load carries it as an immediate; otherwise the table's address is added.
template <bool FIXED, int I>
__device__ __forceinline__ uint32_t lut_byte(uint32_t lut_addr, uint32_t laneword, uint32_t w) {
  const uint32_t off = prmt(laneword, w, 0x1100u | ((4u + I) << 4));
  uint32_t v;
  if (FIXED)
    asm("ld.shared.u32 %0, [%1+65536];" : "=r"(v) : "r"(off));
  else
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(off + lut_addr));
  return v;
}

// Four bytes of w -> four fp16x2 words, from the table or by byte permutes.
template <bool PRMT, bool FIXED>
__device__ __forceinline__ void decode4(uint32_t lut_addr, uint32_t laneword, uint32_t w,
                                        const uint32_t (&lo)[2], const uint32_t (&hi)[2],
                                        uint32_t (&r)[4]) {
  if (PRMT) {
    decode8<0x5140u, 0x7362u>(w, lo, hi, r);
  } else {
    r[0] = lut_byte<FIXED, 0>(lut_addr, laneword, w);
    r[1] = lut_byte<FIXED, 1>(lut_addr, laneword, w);
    r[2] = lut_byte<FIXED, 2>(lut_addr, laneword, w);
    r[3] = lut_byte<FIXED, 3>(lut_addr, laneword, w);
  }
}

__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) {
  return *reinterpret_cast<const uint32_t *>(p);
}

// Table word of a turbo3 sign byte s (element k's high index bit at bit k): the high
// bit of element 2a at bit 4a + 2, that of element 2a + 1 at bit 16 + 4a + 2 -- bit 2
// of nibble a of the two selector words t3_block builds.
__host__ __device__ constexpr uint32_t t3_sign_word(uint32_t s) {
  uint32_t w = 0;
  for (int a = 0; a < 4; ++a)
    w |= (((s >> (2 * a)) & 1u) << (4 * a + 2)) | (((s >> (2 * a + 1)) & 1u) << (16 + 4 * a + 2));
  return w;
}

// Lane t's share of one 32-element turbo3 key block (the "2+1" layout: fp16 norm,
// qs[8] holding the low two index bits of element j at bits 2(j%4) of qs[j/4],
// signs[4] holding its high bit at bit j%8 of signs[j/8]): elements 8t..8t+7, i.e.
// the 16-bit word qs[2t..2t+1] (element 8t+k at bits 2k) and the byte signs[t] (at
// bit k).  The sign byte's bits are spread by one lookup in the key half of the
// table; each 3-bit index then selects a byte of the byte planes lo / hi of the eight
// signed fp16 entries, so any eight-entry codebook decodes.  r gets the fp16x2 pairs
// (e0,e2), (e4,e6), (e1,e3), (e5,e7); returns the block's norm.
template <bool FIXED>
__device__ __forceinline__ float t3_block(const uint8_t *blk, int t, uint32_t lut_addr,
                                          uint32_t laneword, const uint32_t (&lo)[2],
                                          const uint32_t (&hi)[2], uint32_t (&r)[4]) {
  const uint32_t q = *reinterpret_cast<const uint16_t *>(blk + 2 + 2 * t);
  const uint32_t sw = lut_byte<FIXED, 0>(lut_addr, laneword, blk[10 + t]);
  // nibble a of the low half: index of e_2a; of the high half: index of e_2a+1
  const uint32_t x = ((q | (q << 14)) & 0x33333333u) | sw;
  const uint32_t xo = x >> 16;
  const uint32_t le = prmt(lo[0], lo[1], x), he = prmt(hi[0], hi[1], x);
  const uint32_t lodd = prmt(lo[0], lo[1], xo), hodd = prmt(hi[0], hi[1], xo);
  r[0] = prmt(le, he, 0x5140u);
  r[1] = prmt(le, he, 0x7362u);
  r[2] = prmt(lodd, hodd, 0x5140u);
  r[3] = prmt(lodd, hodd, 0x7362u);
  return __half2float(*reinterpret_cast<const __half *>(blk));
}


__device__ __forceinline__ float half_at(const uint8_t *p) {
  return __half2float(*reinterpret_cast<const __half *>(p));
}

// Largest of the four block norms of a 56-byte turbo3 row.
__device__ __forceinline__ float t3_max_norm(const uint8_t *row) {
  return fmaxf(fmaxf(half_at(row), half_at(row + 14)), fmaxf(half_at(row + 28), half_at(row + 42)));
}

// Four 3-bit turbo3 indices, one per byte: byte j = (2-bit field j of the qs byte) | (bit j
// of the sign nibble selected by `shift`) << 2.  The 2-bit fields spread to their bytes by
// two multiplies over disjoint bit ranges (fields 0, 2 by 1 + 2^12; fields 1, 3 by 2^6 +
// 2^18), the four sign bits by one (1 + 2^7 + 2^14 + 2^21).
__device__ __forceinline__ uint32_t t3_index_word(uint32_t qbyte, uint32_t sbyte, uint32_t shift) {
  const uint32_t q = ((qbyte & 0x33u) * 0x1001u & 0x00030003u) | ((qbyte & 0xCCu) * 0x40040u & 0x03000300u);
  const uint32_t sg = ((sbyte >> shift) & 15u) * 0x204081u & 0x01010101u;
  return q | (sg << 2);
}

// The PV B operand of one column group from the probabilities of this lane's two score
// rows: column g takes head g/2, its fp16 hi (g even) or lo (g odd) part, for the keys
// a_t, a_t+2 (k 2t, 2t+1) and a_t+4, a_t+6 (k 2t+8, 2t+9), gathered from the lanes that
// own those keys' scores.
__device__ __forceinline__ void p_operand(float pp0, float pp1, int src0, int src1, float lo_sel,
                                          uint32_t (&pb)[2]) {
  const float va = __shfl_sync(FULL_MASK, pp0, src0), vb = __shfl_sync(FULL_MASK, pp0, src1);
  const float vc = __shfl_sync(FULL_MASK, pp1, src0), vd = __shfl_sync(FULL_MASK, pp1, src1);
  const __half2 hab = __floats2half2_rn(va, vb), hcd = __floats2half2_rn(vc, vd);
  const float2 fab = __half22float2(hab), fcd = __half22float2(hcd);
  const __half2 rab = __floats2half2_rn(fmaf(-lo_sel, fab.x, va), fmaf(-lo_sel, fab.y, vb));
  const __half2 rcd = __floats2half2_rn(fmaf(-lo_sel, fcd.x, vc), fmaf(-lo_sel, fcd.y, vd));
  pb[0] = *reinterpret_cast<const uint32_t *>(&rab);
  pb[1] = *reinterpret_cast<const uint32_t *>(&rcd);
}

// Physical key (within a 16-key block) of score row r.  Rows g and g+8 belong to
// lane group g.  With this order the packed-word loads of a warp hit every bank at
// most twice, and the PV operand of lane (g, t) -- keys a_t, a_t+2, a_t+4, a_t+6
// with a_t = {0, 1, 8, 9}[t] -- comes from score rows t, 4+t, 8+t, 12+t, i.e. from
// the same register of lanes 4t+h and 4(4+t)+h.
__device__ __forceinline__ int key_of_row(int r) {
  // rows 0..7: 0 1 8 9 2 3 10 11; rows 8..15: 4 5 12 13 6 7 14 15
  return ((r & 1) | ((r & 2) << 2) | ((r & 4) >> 1) | ((r & 8) >> 1));
}

// Barrier over the consumer warps only (the producer warp never joins it).
__device__ __forceinline__ void consumers_sync() { named_sync1<CWARPS * 32>(); }

// Persistent split-K decode: one CTA per SM streams its tile range through a ring of
// NSTAGE stages.  Lane (g, t) = (lane / 4, lane % 4) of a consumer warp owns, per
// 16-key block, score rows g and g+8 (head t of every column group) and dims
// 16g..16g+15 of the PV product.  KP of the 4 key words and VP of the 2 value words
// per lane are decoded by byte permutes instead of the table, to balance the ALU and
// shared-memory pipes.
//
// K3: turbo3 keys (56-byte rows of four 32-element blocks, each with its own norm),
// turbo4 values.  The score's k dimension is then ordered block by block: MMA slices
// 2b and 2b+1 cover block b, lane t holding its elements 8t..8t+7 (the q operand is
// permuted to match once per item), and each block's product is scaled by that
// block's norm as it is added to the score.
template <int NG, bool SCORES, int KP, int VP, bool FIXED, bool K3, bool V3>
__global__ void __maxnreg__(128)
    k_partial_t4(const PartialParams p) {
  constexpr int KROW = K3 ? T3_ROW : T4_ROW;
  constexpr int VROW = V3 ? T3_ROW : T4_ROW;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemHead &sm = *reinterpret_cast<SmemHead *>(smem_raw);
  uint32_t *lut = reinterpret_cast<uint32_t *>(smem_raw + LUT_OFF);
  const int cta = blockIdx.x;
  pdl_trigger();
  if (FIXED && smem_addr(smem_raw) != RESERVED_SMEM) {  // layout assumption broken: refuse
    if (threadIdx.x == 0) atomicExch(p.status, (int32_t)DEVERR_LAYOUT);
    return;
  }

  QStage &qst = *reinterpret_cast<QStage *>(smem_raw + QSTAGE_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == CWARPS * 32) {  // the producer's lane sets up the barriers
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], CWARPS);
    }
    mbar_init(&qst.full, 1);
    mbar_init(&qst.empty, CWARPS);
    sm.abort_flag = 0;
    sm.n_units = 0;
    fence_mbar_init();
  }
  if (warp == CWARPS) {
    // ---------------- producer: streams every tile (and every item's q) of the range.  It
    // takes no part in the table fill: once the previous kernel is complete it starts the
    // first copies at once.
    named_arrive0<NTHREADS>();  // the barriers are set up
    if (lane == 0) {
      // The range's first tiles pulled into L2 before the wait on the previous kernel (in a
      // decode loop, while the previous launch merges): a prefetch moves no data into the
      // CTA, and the previous kernel's writes land in L2, so the copies after the wait read
      // current rows.  Units taken at full length (seq_lens may still be written); every
      // range lies inside the rows the copies below read.
      int tp = cta_first_tile(p, cta), n_pre = 0;
      Item ip;
      while (n_pre < PREFETCH_TILES && next_item(p, cta, tp, ip)) {
        const size_t row0 = (size_t)(ip.unit / p.n_hg) * p.L;
        for (int j = ip.t0; j < ip.t1 && n_pre < PREFETCH_TILES && j * TILE < p.L; ++j, ++n_pre) {
          const int nk = min(TILE, p.L - j * TILE);
          const size_t ks = (row0 + (size_t)j * TILE) * KROW, vs = (row0 + (size_t)j * TILE) * VROW;
          const size_t k0 = ks & ~(size_t)15, v0 = vs & ~(size_t)15;
          bulk_prefetch_l2(p.kc + k0, (uint32_t)(((ks + (size_t)nk * KROW + 15) & ~(size_t)15) - k0));
          bulk_prefetch_l2(p.vc + v0, (uint32_t)(((vs + (size_t)nk * VROW + 15) & ~(size_t)15) - v0));
        }
      }
    }
    pdl_wait();
    if (lane == 0) {
      int ctr = 0, tt = cta_first_tile(p, cta), n_item = 0;
      Item it;
      bool ok = true;
      while (ok && next_item(p, cta, tt, it)) {
        // this item's q: after the consumers have taken the previous item's
        if (n_item > 0 && !mbar_wait_bounded(&qst.empty, (n_item - 1) & 1, WAIT_LIMIT_NS)) {
          atomicExch(&sm.abort_flag, 1);
          atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        {
          const int hg = it.unit % p.n_hg, bk = it.unit / p.n_hg;
          const int b = bk / p.Hkv, kvh = bk % p.Hkv;
          const int G = min(4 * NG, p.gq - hg * 4 * NG);
          const size_t row0 = (size_t)b * p.Hq + kvh * p.gq + hg * 4 * NG;
          for (int h = 0; h < G; ++h) qst.qs[h] = p.qsc[2 * (row0 + h)];
          mbar_arrive_expect_tx(&qst.full, (uint32_t)G * 512u);
          for (int h = 0; h < G; ++h) bulk_g2s(qst.q[h], p.qhl + (row0 + h) * 256, 512u, &qst.full);
          ++n_item;
        }
        const int Lb = unit_len(p, it.unit);
        const size_t unit_row0 = (size_t)(it.unit / p.n_hg) * p.L;
        for (int j = it.t0; j < it.t1; ++j) {
          const int kf = j * TILE;
          if (kf >= Lb) break;  // consumers skip the same tiles
          const int nk = min(TILE, Lb - kf);
          const int s = ctr % NSTAGE;
          if (p.withhold_first_tile && ctr == 0) {  // failure test: consumers wait in vain
            ++ctr;
            continue;
          }
          if (ctr >= NSTAGE &&
              !mbar_wait_bounded(&sm.empty[s], ((ctr / NSTAGE) - 1) & 1, WAIT_LIMIT_NS)) {
            atomicExch(&sm.abort_flag, 1);
            atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
            ok = false;
            break;
          }
          const size_t ks = (unit_row0 + kf) * KROW, vs = (unit_row0 + kf) * VROW;
          const size_t k0 = ks & ~(size_t)15, v0 = vs & ~(size_t)15;
          const uint32_t kbytes = (uint32_t)(((ks + (size_t)nk * KROW + 15) & ~(size_t)15) - k0);
          const uint32_t vbytes = (uint32_t)(((vs + (size_t)nk * VROW + 15) & ~(size_t)15) - v0);
          mbar_arrive_expect_tx(&sm.full[s], kbytes + vbytes);
          bulk_g2s(stage_buf(smem_raw, s), p.kc + k0, kbytes, &sm.full[s]);
          bulk_g2s(stage_buf(smem_raw, 4 + s), p.vc + v0, vbytes, &sm.full[s]);
          ++ctr;
        }
      }
      // R for the merge at the CTA's end, pulled into L2 now: the stream has evicted it,
      // and the last few tiles take longer than its fetch
      if (ok && p.out && p.r) bulk_prefetch_l2(p.r, D * D * sizeof(float));
      // Let every issued copy land before the CTA can exit (only matters after a
      // bounded wait gave up; otherwise the consumers have consumed them all).
      if (!ok || sm.abort_flag) {
        for (int c = (ctr > NSTAGE ? ctr - NSTAGE : 0); c < ctr; ++c)
          (void)mbar_wait_bounded(&sm.full[c % NSTAGE], (c / NSTAGE) & 1, WAIT_LIMIT_NS);
        if (n_item > 0) (void)mbar_wait_bounded(&qst.full, (n_item - 1) & 1, WAIT_LIMIT_NS);
      }
    }
    return;
  }
  // Fill the table (consumer warps): each (byte, half) entry is computed once and stored
  // to its 32 slots with 16-byte stores.
  for (int piece = threadIdx.x; piece < 256 * 8; piece += CWARPS * 32) {
    const int byte = piece >> 3, chunk = piece & 7;  // chunks 0-3: key slots, 4-7: value slots
    const uint32_t *c16 = (chunk & 4) ? p.vc16 : p.kc16;
    const uint32_t lo = (c16[(byte & 15) >> 1] >> (16 * (byte & 1))) & 0xFFFFu;
    const uint32_t hi = (c16[(byte >> 4) >> 1] >> (16 * ((byte >> 4) & 1))) & 0xFFFFu;
    // turbo3 values: byte = 3-bit index of key a | 3-bit index of key b << 3 (rows 0-63)
    const uint32_t lo3 = (c16[(byte & 7) >> 1] >> (16 * (byte & 1))) & 0xFFFFu;
    const uint32_t hi3 = (c16[((byte >> 3) & 7) >> 1] >> (16 * ((byte >> 3) & 1))) & 0xFFFFu;
    // turbo3 keys: the key slots hold the spread sign bits instead
    const uint32_t e = (K3 && chunk < 4)   ? t3_sign_word(byte)
                       : (V3 && chunk >= 4) ? (byte < 64 ? lo3 | (hi3 << 16) : 0u)
                                            : lo | (hi << 16);
    uint4 *dst = reinterpret_cast<uint4 *>(lut + byte * 64 + chunk * 8);
    dst[0] = make_uint4(e, e, e, e);
    dst[1] = make_uint4(e, e, e, e);
  }
  pdl_wait();  // the caches, q and the workspace may be written by the previous kernel
  if (threadIdx.x == 0 && p.seq_lens) {
    for (int b = 0; b < p.B; ++b)
      if (p.seq_lens[b] < 1 || p.seq_lens[b] > p.L) atomicExch(p.status, (int32_t)DEVERR_SEQLEN);
  }
  named_sync0<NTHREADS>();  // the table is filled and the barriers are set up
  const int g = lane >> 2, t = lane & 3;

  // ---------------- consumers
  const uint32_t lut_base = smem_addr(lut);
  const uint32_t kword = 4u * lane, vword = 128u + 4u * lane;
  const uint32_t klo[2] = {p.klo[0], p.klo[1]}, khi[2] = {p.khi[0], p.khi[1]};
  const uint32_t vlo[2] = {p.vlo[0], p.vlo[1]}, vhi[2] = {p.vhi[0], p.vhi[1]};
  const int rk0 = key_of_row(g), rk1 = key_of_row(g + 8);
  const int at = (t & 1) | ((t & 2) << 2);  // a_t = 0, 1, 8, 9
  // Tile row of the warp's key k.  Rows 16 apart start 16 banks apart (68-byte rows), so a
  // warp whose keys are rows r0 .. r0+7 and r0+16 .. r0+23 reads its packed words and norms
  // without bank conflicts in every load shape above; warps 0..13 pair up on 32-row blocks
  // that way, and the last warp (and turbo3 keys, whose 56-byte rows differ) keeps 16
  // consecutive rows.  Keys a_t + 2m stay 2m rows after key a_t in both layouts.
  const bool paired = !K3 && !V3 && warp < 2 * (CWARPS / 2);
  const int r0 = paired ? 32 * (warp >> 1) + 8 * (warp & 1) : 16 * warp;
  auto row_of = [&](int k) { return paired ? r0 + (k & 7) + 16 * (k >> 3) : r0 + k; };
  const int pk0 = row_of(rk0), pk1 = row_of(rk1), pat = row_of(at);
  const int hs = g >> 1;
  const int src0 = 4 * t + hs, src1 = 4 * (4 + t) + hs;
  const float lo_sel = (g & 1) ? 1.f : 0.f;

  int ctr = 0, tt = cta_first_tile(p, cta), n_item = 0;
  Item it;
  bool aborted = false;
  // fused combine, thread 0: per recorded unit, b * Hq + its first head and (its head count
  // | its partial count << 4), taken at the item's start, off the merge's path
  int t0_row[FIN_MAX], t0_pk[FIN_MAX];
  while (!aborted && next_item(p, cta, tt, it)) {
    const int Lb = unit_len(p, it.unit);
    const int hg = it.unit % p.n_hg;
    const int bk = it.unit / p.n_hg;
    const int b = bk / p.Hkv, kvh = bk % p.Hkv;
    const int G = min(4 * NG, p.gq - hg * 4 * NG);
    const int head0 = kvh * p.gq + hg * 4 * NG;
    const size_t unit_row0 = (size_t)bk * p.L;
    const int it_nsplit = (p.out && threadIdx.x == 0) ? unit_n_split(p, it.unit) : 0;

    // q as the B operand: column g = (head slot g/2, part g%2 = hi/lo), rows = dims, from
    // the q stage the producer filled for this item
    if (!mbar_wait_bounded(&qst.full, n_item & 1, WAIT_LIMIT_NS)) {
      if (lane == 0) {
        atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
        atomicExch(&sm.abort_flag, 1);
      }
      aborted = true;
      break;
    }
    uint32_t qb[NG][8][2];
    float qs[NG];
#pragma unroll
    for (int c = 0; c < NG; ++c) {
      const int slot = c * 4 + hs;
      if (slot < G && K3) {
        // slice 2b + h, lane t: dims 32b + 8t + 4h + {0, 2} and {1, 3}
        const uint32_t *qw = qst.q[slot] + (g & 1) * 64 + 4 * t;
#pragma unroll
        for (int bl = 0; bl < 4; ++bl) {
          const uint32_t w0 = qw[16 * bl], w1 = qw[16 * bl + 1];
          const uint32_t w2 = qw[16 * bl + 2], w3 = qw[16 * bl + 3];
          qb[c][2 * bl][0] = prmt(w0, w1, 0x5410u);
          qb[c][2 * bl][1] = prmt(w0, w1, 0x7632u);
          qb[c][2 * bl + 1][0] = prmt(w2, w3, 0x5410u);
          qb[c][2 * bl + 1][1] = prmt(w2, w3, 0x7632u);
        }
      } else if (slot < G) {
        const uint32_t *qw = qst.q[slot] + (g & 1) * 64 + 16 * t;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qb[c][kk][0] = qw[2 * kk];
          qb[c][kk][1] = qw[2 * kk + 1];
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) qb[c][kk][0] = qb[c][kk][1] = 0u;
      }
      const int my = c * 4 + t;  // the head whose scores this lane holds
      qs[c] = (my < G) ? qst.qs[my] : 0.f;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&qst.empty);  // this warp's q is in registers
    ++n_item;
    float O[NG][8][4];
    float M[NG], lsum[NG];
#pragma unroll
    for (int c = 0; c < NG; ++c) {
      M[c] = -INFINITY;
      lsum[c] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) O[c][mt][0] = O[c][mt][1] = O[c][mt][2] = O[c][mt][3] = 0.f;
    }

    for (int j = it.t0; j < it.t1; ++j) {
      const int kf = j * TILE;
      if (kf >= Lb) break;
      const int s = ctr % NSTAGE;
      if (!mbar_wait_bounded(&sm.full[s], (ctr / NSTAGE) & 1, WAIT_LIMIT_NS)) {
        if (lane == 0) {
          atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
          atomicExch(&sm.abort_flag, 1);
        }
        aborted = true;
        break;
      }
      const int nk = min(TILE, Lb - kf);
      const size_t ks = (unit_row0 + kf) * KROW, vs = (unit_row0 + kf) * VROW;
      const uint8_t *Ks = stage_buf(smem_raw, s) + (ks & 15);
      const uint8_t *Vs = stage_buf(smem_raw, 4 + s) + (vs & 15);
      if (r0 < nk) {  // the warp's first row is its lowest: some key is valid
        // ---- scores S^T[16 rows x 8 cols] = K_hat Q^T, two accumulator chains
        float sa[NG][4], sb[NG][4];
#pragma unroll
        for (int c = 0; c < NG; ++c)
#pragma unroll
          for (int e = 0; e < 4; ++e) sa[c][e] = sb[c][e] = 0.f;
        if (K3) {
#pragma unroll
          for (int bl = 0; bl < 4; ++bl) {
            uint32_t d0[4], d1[4];
            const float n0 = t3_block<FIXED>(Ks + pk0 * KROW + 14 * bl, t, lut_base, kword, klo, khi, d0);
            const float n1 = t3_block<FIXED>(Ks + pk1 * KROW + 14 * bl, t, lut_base, kword, klo, khi, d1);
            const uint32_t a0[4] = {d0[0], d1[0], d0[2], d1[2]};
            const uint32_t a1[4] = {d0[1], d1[1], d0[3], d1[3]};
#pragma unroll
            for (int c = 0; c < NG; ++c) {
              float acc[4] = {0.f, 0.f, 0.f, 0.f};
              mma_f16(acc, a0, qb[c][2 * bl][0], qb[c][2 * bl][1]);
              mma_f16(acc, a1, qb[c][2 * bl + 1][0], qb[c][2 * bl + 1][1]);
              sa[c][0] = fmaf(n0, acc[0], sa[c][0]);
              sa[c][1] = fmaf(n0, acc[1], sa[c][1]);
              sa[c][2] = fmaf(n1, acc[2], sa[c][2]);
              sa[c][3] = fmaf(n1, acc[3], sa[c][3]);
            }
          }
        }
        const uint8_t *kr0 = Ks + pk0 * KROW + 4 + 16 * t;
        const uint8_t *kr1 = Ks + pk1 * KROW + 4 + 16 * t;
#pragma unroll
        for (int w = 0; w < (K3 ? 0 : 4); ++w) {
          uint32_t d0[4], d1[4];
          const uint32_t x0 = ld_u32(kr0 + 4 * w), x1 = ld_u32(kr1 + 4 * w);
          if (w < KP) {
            decode4<true, FIXED>(lut_base, kword, x0, klo, khi, d0);
            decode4<true, FIXED>(lut_base, kword, x1, klo, khi, d1);
          } else {
            decode4<false, FIXED>(lut_base, kword, x0, klo, khi, d0);
            decode4<false, FIXED>(lut_base, kword, x1, klo, khi, d1);
          }
          const uint32_t a0[4] = {d0[0], d1[0], d0[1], d1[1]};
          const uint32_t a1[4] = {d0[2], d1[2], d0[3], d1[3]};
#pragma unroll
          for (int c = 0; c < NG; ++c) {
            mma_f16(sa[c], a0, qb[c][2 * w][0], qb[c][2 * w][1]);
            mma_f16(sb[c], a1, qb[c][2 * w + 1][0], qb[c][2 * w + 1][1]);
          }
        }
        // ---- online softmax over the two keys of this lane, head t of each group
        // turbo3 keys carry their block norms in sa already
        const float nk0 = K3 ? 1.f : *reinterpret_cast<const float *>(Ks + pk0 * KROW);
        const float nk1 = K3 ? 1.f : *reinterpret_cast<const float *>(Ks + pk1 * KROW);
        // turbo3 values: the largest of the key's four block norms goes into the exponent,
        // each block's ratio to it into that block's probability operand
        const float nv0 = V3 ? t3_max_norm(Vs + pk0 * VROW) : *reinterpret_cast<const float *>(Vs + pk0 * VROW);
        const float nv1 = V3 ? t3_max_norm(Vs + pk1 * VROW) : *reinterpret_cast<const float *>(Vs + pk1 * VROW);
        const bool ok0 = pk0 < nk, ok1 = pk1 < nk;
        const float nu0 = ok0 ? fmaxf(log2_approx(nv0), -64.f) : 0.f;
        const float nu1 = ok1 ? fmaxf(log2_approx(nv1), -64.f) : 0.f;
        uint32_t pb[NG][2];
        float pq0[NG], pq1[NG];  // turbo3 values: the probabilities, scaled per block below
#pragma unroll
        for (int c = 0; c < NG; ++c) {
          const float d0 = K3 ? sa[c][0] + sa[c][1] : (sa[c][0] + sa[c][1]) + (sb[c][0] + sb[c][1]);
          const float d1 = K3 ? sa[c][2] + sa[c][3] : (sa[c][2] + sa[c][3]) + (sb[c][2] + sb[c][3]);
          const float s0 = ok0 ? d0 * (nk0 * qs[c]) : -INFINITY;
          const float s1 = ok1 ? d1 * (nk1 * qs[c]) : -INFINITY;
          if (SCORES && c * 4 + t < G) {
            float *srow = p.scores + (size_t)(b * p.Hq + head0 + c * 4 + t) * p.L + kf;
            if (ok0) srow[pk0] = s0 * LN2;
            if (ok1) srow[pk1] = s1 * LN2;
          }
          const float u0 = s0 + nu0, u1 = s1 + nu1;
          float bm = fmaxf(u0, u1);
          bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 4));
          bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 8));
          bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 16));
          if (bm > M[c] + RESCALE_SLACK) {  // also taken while M is -inf
            const float alpha = exp2_approx(M[c] - bm);
            M[c] = bm;
            lsum[c] *= alpha;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              O[c][mt][0] *= alpha, O[c][mt][1] *= alpha, O[c][mt][2] *= alpha, O[c][mt][3] *= alpha;
            }
          }
          const float Mu = (M[c] == -INFINITY) ? 0.f : M[c];
          lsum[c] += exp2_approx(s0 - Mu) + exp2_approx(s1 - Mu);
          const float pp0 = exp2_approx(u0 - Mu + P_SHIFT);
          const float pp1 = exp2_approx(u1 - Mu + P_SHIFT);
          if (V3) {
            pq0[c] = pp0, pq1[c] = pp1;
          } else {
            p_operand(pp0, pp1, src0, src1, lo_sel, pb[c]);
          }
        }
        if (V3) {
          // ---- turbo3 values.  Each 16-row m-tile lies inside one 32-element block b: m-tile
          // 2b + h, rows g and g+8 = elements 4g + 2h and 4g + 2h + 1 of block b, so block b's
          // norm (over the key's largest, which sits in the exponent) scales that m-tile's
          // probability operand exactly; lane group g decodes elements 4g .. 4g+3 of every
          // block, two keys per table lookup (a 6-bit index: 3 bits of each key).
          // (rows past the tile's valid keys hold stale bytes: their ratios are forced to 0)
          const float inv0 = (ok0 && nv0 > 0.f) ? 1.f / nv0 : 0.f, inv1 = (ok1 && nv1 > 0.f) ? 1.f / nv1 : 0.f;
          const uint8_t *vq = Vs + pat * VROW + 2 + g;            // key a_t, block 0: qs byte g
          const uint8_t *vsg = Vs + pat * VROW + 10 + (g >> 1);  // and its sign byte
          const uint32_t ssh = 4u * (g & 1);
#pragma unroll
          for (int bl = 0; bl < 4; ++bl) {
            const float r0 = inv0 > 0.f ? half_at(Vs + pk0 * VROW + 14 * bl) * inv0 : 0.f;
            const float r1 = inv1 > 0.f ? half_at(Vs + pk1 * VROW + 14 * bl) * inv1 : 0.f;
            uint32_t pbb[NG][2];
#pragma unroll
            for (int c = 0; c < NG; ++c) p_operand(pq0[c] * r0, pq1[c] * r1, src0, src1, lo_sel, pbb[c]);
            uint32_t wk[4];  // keys a_t + 2i: byte j = 3-bit index of element 4g + j
#pragma unroll
            for (int i = 0; i < 4; ++i)
              wk[i] = t3_index_word(vq[2 * i * VROW + 14 * bl], vsg[2 * i * VROW + 14 * bl], ssh);
            const uint32_t w01 = wk[0] | (wk[1] << 3), w23 = wk[2] | (wk[3] << 3);
            {
              const uint32_t a[4] = {lut_byte<FIXED, 0>(lut_base, vword, w01), lut_byte<FIXED, 1>(lut_base, vword, w01),
                                     lut_byte<FIXED, 0>(lut_base, vword, w23), lut_byte<FIXED, 1>(lut_base, vword, w23)};
#pragma unroll
              for (int c = 0; c < NG; ++c) mma_f16(O[c][2 * bl], a, pbb[c][0], pbb[c][1]);
            }
            {
              const uint32_t a[4] = {lut_byte<FIXED, 2>(lut_base, vword, w01), lut_byte<FIXED, 3>(lut_base, vword, w01),
                                     lut_byte<FIXED, 2>(lut_base, vword, w23), lut_byte<FIXED, 3>(lut_base, vword, w23)};
#pragma unroll
              for (int c = 0; c < NG; ++c) mma_f16(O[c][2 * bl + 1], a, pbb[c][0], pbb[c][1]);
            }
          }
        }
        // ---- O^T[dims x cols] += V_hat^T[dims x keys] P^T
        const uint8_t *va_p = Vs + pat * VROW + 4 + 8 * g;  // key a_t; a_t+2, +4, +6 follow
#pragma unroll
        for (int w = 0; w < (V3 ? 0 : 2); ++w) {
          const uint32_t xa = ld_u32(va_p + 4 * w), xb = ld_u32(va_p + 2 * T4_ROW + 4 * w);
          const uint32_t xc = ld_u32(va_p + 4 * T4_ROW + 4 * w), xd = ld_u32(va_p + 6 * T4_ROW + 4 * w);
          // byte i of zlo = (low nibble of key a, low nibble of key b) of byte 8g + 4w + i
          const uint32_t zlo_ab = (xa & 0x0F0F0F0Fu) | ((xb << 4) & 0xF0F0F0F0u);
          const uint32_t zhi_ab = ((xa >> 4) & 0x0F0F0F0Fu) | (xb & 0xF0F0F0F0u);
          const uint32_t zlo_cd = (xc & 0x0F0F0F0Fu) | ((xd << 4) & 0xF0F0F0F0u);
          const uint32_t zhi_cd = ((xc >> 4) & 0x0F0F0F0Fu) | (xd & 0xF0F0F0F0u);
          uint32_t r0[4], r1[4], r2[4], r3[4];
          if (w < VP) {
            decode4<true, FIXED>(lut_base, vword, zlo_ab, vlo, vhi, r0);
            decode4<true, FIXED>(lut_base, vword, zhi_ab, vlo, vhi, r1);
            decode4<true, FIXED>(lut_base, vword, zlo_cd, vlo, vhi, r2);
            decode4<true, FIXED>(lut_base, vword, zhi_cd, vlo, vhi, r3);
          } else {
            decode4<false, FIXED>(lut_base, vword, zlo_ab, vlo, vhi, r0);
            decode4<false, FIXED>(lut_base, vword, zhi_ab, vlo, vhi, r1);
            decode4<false, FIXED>(lut_base, vword, zlo_cd, vlo, vhi, r2);
            decode4<false, FIXED>(lut_base, vword, zhi_cd, vlo, vhi, r3);
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint32_t a[4] = {r0[jj], r1[jj], r2[jj], r3[jj]};
#pragma unroll
            for (int c = 0; c < NG; ++c) mma_f16(O[c][4 * w + jj], a, pb[c][0], pb[c][1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
      ++ctr;
    }
    // A warp that gave up waiting has set the flag before any warp can get here past
    // the same tile, so either every consumer warp enters the merge barriers or none.
    if (aborted || *reinterpret_cast<volatile int *>(&sm.abort_flag)) break;
#pragma unroll
    for (int c = 0; c < NG; ++c) {
      lsum[c] += __shfl_xor_sync(FULL_MASK, lsum[c], 4);
      lsum[c] += __shfl_xor_sync(FULL_MASK, lsum[c], 8);
      lsum[c] += __shfl_xor_sync(FULL_MASK, lsum[c], 16);
    }

    // ---- merge the consumer warps' states of this item and write its partial
    if (g == 0) {
#pragma unroll
      for (int c = 0; c < NG; ++c) {
        sm.mw[warp][c * 4 + t] = M[c];
        sm.lw[warp][c * 4 + t] = lsum[c];
      }
    }
    consumers_sync();
#pragma unroll
    for (int c = 0; c < NG; ++c) {
      const int hh = c * 4 + t;
      // the head's max and sum over the warps, by shuffles: lane (g, t) takes warps g and
      // g + 8, the xor steps over g combine them (every lane of a warp ends with its t's)
      const float m0 = sm.mw[g][hh], l0 = sm.lw[g][hh];
      const bool has1 = g + 8 < CWARPS;
      const float m1 = has1 ? sm.mw[g + 8][hh] : -INFINITY, l1 = has1 ? sm.lw[g + 8][hh] : 0.f;
      float ms = fmaxf(m0, m1);
      ms = fmaxf(ms, __shfl_xor_sync(FULL_MASK, ms, 4));
      ms = fmaxf(ms, __shfl_xor_sync(FULL_MASK, ms, 8));
      ms = fmaxf(ms, __shfl_xor_sync(FULL_MASK, ms, 16));
      float ls = (m0 == -INFINITY ? 0.f : l0 * exp2_approx(m0 - ms)) +
                 (m1 == -INFINITY ? 0.f : l1 * exp2_approx(m1 - ms));
      ls += __shfl_xor_sync(FULL_MASK, ls, 4);
      ls += __shfl_xor_sync(FULL_MASK, ls, 8);
      ls += __shfl_xor_sync(FULL_MASK, ls, 16);
      const float fac = (M[c] == -INFINITY) ? 0.f : exp2_approx(M[c] - ms);
      // rows g and g+8 of m-tile mt: dims 16g + 2mt and +1 (turbo4 values), or for turbo3
      // values (m-tile 2b + h inside block b) dims 32b + 4g + 2h and +1
      float *orow = &sm.osm[warp][t][0];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int dm = V3 ? 32 * (mt >> 1) + 4 * g + 2 * (mt & 1) : 16 * g + 2 * mt;
        orow[dm] = (O[c][mt][0] + O[c][mt][1]) * fac;
        orow[dm + 1] = (O[c][mt][2] + O[c][mt][3]) * fac;
      }
      consumers_sync();
      const int Gc = min(4, G - c * 4);
      for (int idx = threadIdx.x; idx < Gc * D; idx += CWARPS * 32) {
        const int h4 = idx / D, jd = idx % D;
        const int hh2 = c * 4 + h4;
        // (warp-uniform h4: lane h4 = (g 0, t h4) holds that head's max and sum)
        const float ms2 = __shfl_sync(FULL_MASK, ms, h4), ls2 = __shfl_sync(FULL_MASK, ls, h4);
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < CWARPS; ++w) acc += sm.osm[w][h4][jd];
        float *dst = p.part + ((size_t)(b * p.Hq + head0 + hh2) * p.n_part + it.slot) * PARTIAL_FLOATS;
        dst[6 + jd] = (ms2 == -INFINITY) ? 0.f : acc;
        if (jd < 6) dst[jd] = jd == 0 ? ms2 : (jd == 1 ? ls2 : 0.f);
      }
      consumers_sync();
    }
    // fused combine: the unit's count is raised once at the CTA's end, for all its items
    if (p.out && threadIdx.x == 0) {
      if (sm.n_units < FIN_MAX) {
        const int n = sm.n_units++;
        sm.units[n] = it.unit;
        t0_row[n] = b * p.Hq + head0;
        t0_pk[n] = G | (it_nsplit << 4);
      } else {  // (the host launches the fused form only where a CTA meets at most FIN_MAX units)
        atomicExch(p.status, (int32_t)DEVERR_LAYOUT);
      }
    }
  }

  // ---------------- fused combine of the units this CTA completed: merge every CTA's
  // partial (m* = max m_s, l* = sum l_s 2^(m_s - m*), o = sum acc_s 2^(m_s - m*) / l*), then
  // out = R^T o with R staged in the stage buffers, which are idle now (every copy was
  // consumed).  Only after a clean finish: a CTA that gave up leaves its units unwritten
  // and the status flag set.
  if (!p.out) return;
  // R is copied into the idle stage buffers at once, by every CTA that finished cleanly
  // (every tile was consumed: the last item ended with a barrier of all consumer warps;
  // no warp can give up after that), so that it lands while the counts make their
  // round trip; most CTAs complete a unit.
  float *rs = reinterpret_cast<float *>(smem_raw + STAGE_B_OFF);  // R, row-major [128][128]
  static_assert(6 * STAGE_BUF >= D * D * 4, "R fits in the idle stage buffers");
  const bool r_copy = p.r && !*reinterpret_cast<volatile int *>(&sm.abort_flag);
  if (r_copy) {
    for (int i = threadIdx.x; i < D * D / 4; i += CWARPS * 32)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(rs + 4 * i)), "l"(p.r + 4 * i)
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  // The completed units' rows and (head count | partial count << 4), by thread 0 into the
  // idle stage buffer A (no copy is in flight after a clean finish).
  int *meta = reinterpret_cast<int *>(smem_raw + STAGE_A_OFF);
  // Every consumer thread's partial stores fenced, then one count per item; the CTA whose
  // count completes a unit merges it.  The atomics are issued together (one round trip).
  __threadfence();
  consumers_sync();
  // (the flag, read after the barrier, is the same for every consumer warp)
  const bool gave_up = *reinterpret_cast<volatile int *>(&sm.abort_flag);
  if (threadIdx.x == 0 && !gave_up) {
    const int ni = sm.n_units;
    int old[FIN_MAX];
#pragma unroll
    for (int i = 0; i < FIN_MAX; ++i) old[i] = i < ni ? atomicAdd(&p.unit_done[sm.units[i]], 1) : -1;
    int nf = 0;  // completed units, compacted in place
#pragma unroll
    for (int i = 0; i < FIN_MAX; ++i)
      if (i < ni && old[i] == (t0_pk[i] >> 4) - 1) {
        sm.units[nf] = sm.units[i], meta[nf] = t0_row[i], meta[FIN_MAX + nf] = t0_pk[i];
        ++nf;
      }
    sm.n_units = nf;
    __threadfence();  // the other CTAs' partials, published before their counts
  }
  consumers_sync();
  const int n_fin = gave_up ? 0 : sm.n_units;
  if (n_fin == 0) {
    if (r_copy) asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }
  // The completed units' heads in quads of four (NG quads per unit), up to three quads per
  // pass: the pass's nh heads are merged by twelve warps (W = 12 / nh per head, see
  // below), and thread (quad, j) un-rotates dim j of that quad's heads, with R from the
  // stage buffers (its copy was issued before the counts).
  constexpr int QUADS = 3;
  static_assert(4 * QUADS <= CWARPS && QUADS * D <= CWARPS * 32, "a round's heads and dims");
  const int n_quads = n_fin * NG;
  for (int q0 = 0; q0 < n_quads; q0 += QUADS) {
    // nh heads in this pass; W warps per head split its partials between them (warp w takes
    // head slot w % nh and every W-th chunk of eight splits from chunk w / nh)
    // (nq = 1: four heads, W = 3; nq = 2 or 3: eight or twelve heads, W = 1)
    const int nq = min(QUADS, n_quads - q0), nh = 4 * nq, W = nq == 1 ? 3 : 1;
    const int hs = nq == 1 ? (warp & 3) : warp, part = nq == 1 ? (warp >> 2) : (warp < nh ? 0 : 1);
    if (part < W) {
      const int qq = q0 + (hs >> 2);
      const int ui = qq / NG;  // the completed unit
      const int G = meta[FIN_MAX + ui] & 15;
      const int hu = 4 * (qq % NG) + (hs & 3);  // head within the unit
      float ms = -INFINITY, lsum = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};  // lane l: dims l + 32 m
      if (hu < G) {
        const int n_split = meta[FIN_MAX + ui] >> 4;
        const float *part_base = p.part + (size_t)(meta[ui] + hu) * p.n_part * PARTIAL_FLOATS;
        for (int s0 = 8 * part; s0 < n_split; s0 += 8 * W) {
          // eight splits' (max, sum) and accumulator slices loaded at once
          float mh[8], lh[8], v[8][4];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float *ps = part_base + (size_t)min(s0 + i, n_split - 1) * PARTIAL_FLOATS;
            mh[i] = __ldcg(ps), lh[i] = __ldcg(ps + 1);
#pragma unroll
            for (int m = 0; m < 4; ++m) v[i][m] = __ldcg(ps + 6 + lane + 32 * m);
          }
          // running merge: raise the max of this chunk's live splits, rescale what is held
          float mc = -INFINITY;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (s0 + i < n_split && lh[i] > 0.f) mc = fmaxf(mc, mh[i]);
          if (mc > ms) {
            const float a = (ms == -INFINITY) ? 0.f : exp2f(ms - mc);
            lsum *= a;
#pragma unroll
            for (int m = 0; m < 4; ++m) acc[m] *= a;
            ms = mc;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (s0 + i < n_split && lh[i] > 0.f) {
              const float w = exp2f(mh[i] - ms);
              lsum += w * lh[i];
#pragma unroll
              for (int m = 0; m < 4; ++m) acc[m] = fmaf(w, v[i][m], acc[m]);
            }
          }
        }
      }
      // this warp's share of the head: (max, sum) and its unnormalised accumulator
      if (lane == 0) sm.mw[warp][0] = ms, sm.lw[warp][0] = lsum;
#pragma unroll
      for (int m = 0; m < 4; ++m) sm.osm[warp][1][lane + 32 * m] = acc[m];
    }
    consumers_sync();
    if (warp < nh) {  // the W shares of head slot `warp`, merged (heads past G unused)
      float mx = -INFINITY;
      for (int pp = 0; pp < W; ++pp) mx = fmaxf(mx, sm.mw[warp + pp * nh][0]);
      float lt = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
      for (int pp = 0; pp < W; ++pp) {
        const int w2 = warp + pp * nh;
        const float m2 = sm.mw[w2][0];
        if (m2 != -INFINITY) {
          const float f = exp2f(m2 - mx);
          lt += f * sm.lw[w2][0];
#pragma unroll
          for (int m = 0; m < 4; ++m) o[m] = fmaf(f, sm.osm[w2][1][lane + 32 * m], o[m]);
        }
      }
      const float fo = lt > 0.f ? p.inv_vscale / lt : 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) sm.osm[warp][0][lane + 32 * m] = o[m] * fo;
    }
    if (q0 == 0 && r_copy) asm volatile("cp.async.wait_all;" ::: "memory");
    consumers_sync();  // merged heads (and, the first time, R) in shared memory
    // out = R^T o: thread (group, j) reads column j of R once for the four heads of a quad
    // (o read as broadcast float4), four independent chains over k per head, summed at the
    // end.  With three quads in the pass each group takes one; with one quad the three
    // groups split k in three (the partial sums of groups 1 and 2 meet in the shares'
    // scratch, idle now); with two quads each group takes one.
    const int ks = (nq == 1 && p.r) ? 3 : 1;  // uniform over the CTA
    const int grp = threadIdx.x / D, j = threadIdx.x % D;
    const int qs = ks == 1 ? grp : 0, kpart = ks == 1 ? 0 : grp;
    const int qq = q0 + qs;
    const bool act = grp < QUADS && qs < nq;
    float res[4];
    if (act) {
      const int hb = 4 * qs;
      if (p.r) {
        const int kb = 44 * kpart, ke = ks == 1 ? D : min(D, kb + 44);
        float c4[4][4];
#pragma unroll
        for (int h = 0; h < 4; ++h) c4[h][0] = c4[h][1] = c4[h][2] = c4[h][3] = 0.f;
#pragma unroll 4
        for (int k = kb; k < ke; k += 4) {
          const float r0 = rs[k * D + j], r1 = rs[(k + 1) * D + j];
          const float r2 = rs[(k + 2) * D + j], r3 = rs[(k + 3) * D + j];
#pragma unroll
          for (int h = 0; h < 4; ++h) {  // heads past G hold stale values and are not stored
            const float4 o4 = *reinterpret_cast<const float4 *>(&sm.osm[hb + h][0][k]);
            c4[h][0] = fmaf(r0, o4.x, c4[h][0]);
            c4[h][1] = fmaf(r1, o4.y, c4[h][1]);
            c4[h][2] = fmaf(r2, o4.z, c4[h][2]);
            c4[h][3] = fmaf(r3, o4.w, c4[h][3]);
          }
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) res[h] = (c4[h][0] + c4[h][1]) + (c4[h][2] + c4[h][3]);
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h) res[h] = sm.osm[hb + h][0][j];
      }
      if (kpart > 0) {
#pragma unroll
        for (int h = 0; h < 4; ++h) sm.osm[4 * kpart + h][1][j] = res[h];
      }
    }
    if (ks > 1) consumers_sync();  // the k parts of groups 1 and 2 in shared memory
    if (act && kpart == 0) {
      if (ks > 1) {
#pragma unroll
        for (int h = 0; h < 4; ++h) res[h] += sm.osm[4 + h][1][j] + sm.osm[8 + h][1][j];
      }
      const int ui = qq / NG, G = meta[FIN_MAX + ui] & 15;
      const int hu0 = 4 * (qq % NG);  // first head of the quad within the unit
      float *dst = p.out + (size_t)(meta[ui] + hu0) * D + j;
#pragma unroll
      for (int h = 0; h < 4; ++h)
        if (hu0 + h < G) dst[h * D] = res[h];
    }
    consumers_sync();  // the pass's merged heads are free again
  }
  if (threadIdx.x < n_fin) p.unit_done[sm.units[threadIdx.x]] = 0;
}

struct CombineParams {
  const float *part;
  int n_heads;      // B * Hq (decode) or B * T * Hq (prefill rows)
  int n_split;      // partial slots per head
  int Hq, gq, heads_per_cta, n_hg, tiles_per_unit, sched_g, sched_v, vx;
  uint32_t sched_q, sched_r;  // V / G and V % G (set_schedule)
  float sched_ginv, sched_inv;  // 1 / G and G / V
  int pf_T, pf_Hkv, pf_qpt, pf_n_qt;  // prefill geometry (pf_T = 0: decode)
  int no_main;      // 1: no split-K partials (every key is in the exact tail)
  int tail_slot;    // slot of an exact-tail partial per head, or -1
  const float *r;   // R (row-major) of the value rotation, or null
  float inv_vscale; // 1 / (2^P_SHIFT * alpha_V)
  float *out;
};

// Merge the splits of 8 heads per CTA (one warp each): m* = max m_s,
// l* = sum l_s 2^(m_s - m*), o = sum acc_s 2^(m_s - m*) / l*, then out = R^T o with R
// staged once per CTA.
__global__ void __launch_bounds__(QWARPS * 32) k_combine(const CombineParams p) {
  extern __shared__ __align__(16) float csm[];
  float *r = csm;              // [128][128]
  float *o = csm + D * D;      // [QWARPS][128]
  pdl_trigger();
  if (p.r) stage_matrix(r, p.r);
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x * QWARPS + warp;
  const bool live = bh < p.n_heads;
  if (live) {
    const float *part = p.part + (size_t)bh * p.n_split * PARTIAL_FLOATS;
    // slots written for this head: CTAs whose tile range meets its unit
    int unit;
    if (p.pf_T) {  // row (b, i, h) of a prefill: unit (b, KV head, query tile)
      const int h = bh % p.Hq, i = (bh / p.Hq) % p.pf_T, b = bh / (p.Hq * p.pf_T);
      unit = (b * p.pf_Hkv + h / p.gq) * p.pf_n_qt + i / p.pf_qpt;
    } else {
      const int b = bh / p.Hq, h = bh % p.Hq;
      unit = (b * (p.Hq / p.gq) + h / p.gq) * p.n_hg + (h % p.gq) / p.heads_per_cta;
    }
    const int n_main = p.no_main ? 0 : unit_n_split(p, unit);
    const int n_split = n_main + (p.tail_slot >= 0 ? 1 : 0);
    auto slot = [&](int s) { return s < n_main ? s : p.tail_slot; };  // the tail partial last
    float ms = -INFINITY;
    for (int s = lane; s < n_split; s += 32) {
      const float *ps = part + (size_t)slot(s) * PARTIAL_FLOATS;
      if (ps[1] > 0.f) ms = fmaxf(ms, ps[0]);
    }
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1) ms = fmaxf(ms, __shfl_xor_sync(FULL_MASK, ms, h));
    float lsum = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < n_split; s0 += 32) {
      const int s = s0 + lane;
      float w = 0.f;
      if (s < n_split) {
        const float *ps = part + (size_t)slot(s) * PARTIAL_FLOATS;
        if (ps[1] > 0.f) {
          w = exp2f(ps[0] - ms);
          lsum += w * ps[1];
        }
      }
      const int n = min(32, n_split - s0);
      for (int i0 = 0; i0 < n; i0 += 8) {  // eight splits' loads in flight at a time
        float v[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int si = min(s0 + i0 + i, n_split - 1);
          const float *ps = part + (size_t)slot(si) * PARTIAL_FLOATS + 6;
#pragma unroll
          for (int m = 0; m < 4; ++m) v[i][m] = ps[lane + 32 * m];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float wi = __shfl_sync(FULL_MASK, w, (i0 + i) & 31);
          if (i0 + i < n) {
#pragma unroll
            for (int m = 0; m < 4; ++m) acc[m] = fmaf(wi, v[i][m], acc[m]);
          }
        }
      }
    }
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1) lsum += __shfl_xor_sync(FULL_MASK, lsum, h);
    const float f = p.inv_vscale / lsum;
#pragma unroll
    for (int m = 0; m < 4; ++m) o[warp * D + lane + 32 * m] = acc[m] * f;
  }
  __syncthreads();
  if (!live) return;
  float res[4];
  if (p.r) {
    res[0] = res[1] = res[2] = res[3] = 0.f;
#pragma unroll 8
    for (int k = 0; k < D; ++k) {
      const float ok = o[warp * D + k];
      const float *row = r + k * D + lane;  // (R^T o)_j = sum_k R[k][j] o_k
#pragma unroll
      for (int m = 0; m < 4; ++m) res[m] = fmaf(row[32 * m], ok, res[m]);
    }
  } else {
#pragma unroll
    for (int m = 0; m < 4; ++m) res[m] = o[warp * D + lane + 32 * m];
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) p.out[(size_t)bh * D + lane + 32 * m] = res[m];
}

}  // namespace

bool decode_shape(const tq_ctx *k, const tq_ctx *v, int B, int Hq, int Hkv, int L,
                  DecodeShape *s) {
  s->B = B, s->Hq = Hq, s->Hkv = Hkv, s->L = L;
  s->gq = Hq / Hkv;
  s->pv = k->fmt == TQ_FMT_PROD3;
  s->tile = s->pv ? PV_TILE : T4_TILE;
  s->heads_per_cta = (s->pv || s->gq > 4) ? 8 : 4;
  s->n_hg = (s->gq + s->heads_per_cta - 1) / s->heads_per_cta;
  const int64_t units = (int64_t)B * Hkv * s->n_hg;
  s->tiles_per_unit = (L + s->tile - 1) / s->tile;
  const int64_t total = units * s->tiles_per_unit;
  s->vx = s->pv ? PV_ITEM_TILES
                : (k->fmt == TQ_FMT_TURBO3 || v->fmt == TQ_FMT_TURBO3) ? T3_ITEM_TILES : T4_ITEM_TILES;
  const int64_t vtotal = units * (s->vx + s->tiles_per_unit);
  if (vtotal > INT32_MAX) return false;
  s->total_tiles = (int)total;
  // One persistent CTA per SM; the virtual tile sequence (each unit with its item cost
  // ahead of its tiles) split in proportion, so the ranges differ by at most one tile.
  s->vtotal = (int)vtotal;
  s->grid = (int)(vtotal < k->num_sms ? vtotal : k->num_sms);
  const int shortest = (int)(vtotal / s->grid);
  s->tiles_per_cta = (int)((vtotal + s->grid - 1) / s->grid);
  // Partial slots per head: CTAs whose range meets one unit.
  s->n_part = (s->tiles_per_unit + shortest - 1) / shortest + 1;
  return true;
}

Workspace carve_workspace(const DecodeShape &s, void *base) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t nq = (size_t)s.B * s.Hq;
  const size_t b_qhl = up(nq * 256 * sizeof(uint32_t));
  const size_t b_qsc = up(nq * 2 * sizeof(float));
  const size_t b_part = up(nq * s.n_part * PARTIAL_FLOATS * sizeof(float));
  const int n_units = s.B * s.Hkv * (s.n_hg > 0 ? s.n_hg : 1);
  const size_t b_cnt = up((size_t)n_units * sizeof(int32_t));
  Workspace w{};
  uint8_t *p = static_cast<uint8_t *>(base);
  w.qhl = reinterpret_cast<uint32_t *>(p);
  w.qsc = reinterpret_cast<float *>(p ? p + b_qhl : nullptr);
  w.partials = reinterpret_cast<float *>(p ? p + b_qhl + b_qsc : nullptr);
  w.unit_done = reinterpret_cast<int32_t *>(p ? p + b_qhl + b_qsc + b_part : nullptr);
  w.n_units = n_units;
  w.bytes = b_qhl + b_qsc + b_part + b_cnt;
  return w;
}

QprepParams make_qprep_params(const tq_ctx *k, const void *q, int q_dtype, const DecodeShape &s,
                              float scale, const Workspace &ws) {
  QprepParams p{};
  p.q = q;
  p.q_dtype = q_dtype;
  p.n_q = s.B * s.Hq;
  p.r = k->d_pi;
  p.s = s.pv ? k->d_S : nullptr;
  p.mul = LOG2E * scale / k->f16.alpha;
  p.mul_sk = (float)(LOG2E * (double)scale * (double)k->qjl_factor * 1.2533141373155003 / D);  // sqrt(pi/2) / d
  p.qhl = ws.qhl;
  p.qsc = ws.qsc;
  p.unit_done = ws.unit_done;
  p.n_units = ws.n_units;
  return p;
}

cudaError_t launch_prepare_q(const tq_ctx *k, const void *q, int q_dtype, const DecodeShape &s,
                             float scale, const Workspace &ws, cudaStream_t st) {
  const QprepParams p = make_qprep_params(k, q, q_dtype, s, scale, ws);
  const int grid = (p.n_q + QWARPS - 1) / QWARPS;
  auto kern = s.pv ? k_prepare_q<true> : k_prepare_q<false>;
  cudaError_t e = kernel_smem_attr((const void *)kern, (int)QPREP_SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(QWARPS * 32), QPREP_SMEM, st, p);
}

template <int NG, bool SC, int KP, int VP, bool FIXED, bool K3, bool V3>
cudaError_t launch_t4(const PartialParams &p, dim3 grid, cudaStream_t st) {
  const size_t smem = SMEM_BYTES;
  auto kern = k_partial_t4<NG, SC, KP, VP, FIXED, K3, V3>;
  cudaError_t e = kernel_smem_attr((const void *)kern, (int)smem, true);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(NTHREADS), smem, st, p);
}

// Decode-word split between the table (shared-memory pipe) and byte permutes (ALU pipe):
// of the 4 key words and 2 value words a lane decodes per 16-key block.
constexpr int K_PRMT_WORDS = 0;
constexpr int V_PRMT_WORDS = 0;

template <bool K3, bool V3>
cudaError_t launch_t4_variant(const PartialParams &p, int heads_per_cta, bool fixed, bool scores,
                              dim3 grid, cudaStream_t st) {
  constexpr int KP = K3 ? 0 : K_PRMT_WORDS;
  constexpr int VP = V3 ? 0 : V_PRMT_WORDS;
  if (heads_per_cta == 8) {
    if (fixed)
      return scores ? launch_t4<2, true, KP, VP, true, K3, V3>(p, grid, st)
                    : launch_t4<2, false, KP, VP, true, K3, V3>(p, grid, st);
    return scores ? launch_t4<2, true, KP, VP, false, K3, V3>(p, grid, st)
                  : launch_t4<2, false, KP, VP, false, K3, V3>(p, grid, st);
  }
  if (fixed)
    return scores ? launch_t4<1, true, KP, VP, true, K3, V3>(p, grid, st)
                  : launch_t4<1, false, KP, VP, true, K3, V3>(p, grid, st);
  return scores ? launch_t4<1, true, KP, VP, false, K3, V3>(p, grid, st)
                : launch_t4<1, false, KP, VP, false, K3, V3>(p, grid, st);
}

// The fused combine serves the plain turbo4 / turbo3-key decode (no exact tail) when a CTA
// completes at most FIN_MAX units: it touches at most tiles_per_cta / (vx + tiles_per_unit) + 2.
bool partial_fuses_combine(const DecodeShape &s) {
  return !s.pv && s.tail_slot < 0 && !s.no_main && s.tiles_per_cta / (s.vx + s.tiles_per_unit) + 2 <= FIN_MAX;
}

cudaError_t launch_partial(const tq_ctx *k, const tq_ctx *v, const uint8_t *kc,
                           const uint8_t *vc, const int32_t *seq_lens, const DecodeShape &s,
                           float *scores_dbg, const Workspace &ws, cudaStream_t st,
                           bool withhold_first_tile, float *out, bool *fused) {
  if (fused) *fused = false;
  if (s.pv) return launch_partial_pv(k, v, kc, vc, seq_lens, s, scores_dbg, ws, st);
  PartialParams p{};
  const bool fuse = out && ws.unit_done && partial_fuses_combine(s);
  if (fuse) {
    p.out = out;
    p.r = v->d_pi;
    p.inv_vscale = 1.0f / (exp2f(P_SHIFT) * v->f16.alpha);
    p.unit_done = ws.unit_done;
  }
  p.withhold_first_tile = withhold_first_tile ? 1 : 0;
  p.kc = kc, p.vc = vc, p.seq_lens = seq_lens;
  p.B = s.B, p.Hq = s.Hq, p.Hkv = s.Hkv, p.L = s.L, p.gq = s.gq, p.n_hg = s.n_hg;
  p.tiles_per_unit = s.tiles_per_unit, p.vx = s.vx;
  if (!set_schedule(p, s.grid, s.vtotal)) return cudaErrorInvalidValue;
  p.total_tiles = s.total_tiles, p.n_part = s.n_part;
  p.qhl = ws.qhl, p.qsc = ws.qsc, p.part = ws.partials, p.scores = scores_dbg;
  const bool k3 = k->fmt == TQ_FMT_TURBO3;
  for (int i = 0; i < 2; ++i) {
    p.klo[i] = k->f16.lo[i], p.khi[i] = k->f16.hi[i];
    p.vlo[i] = v->f16.lo[i], p.vhi[i] = v->f16.hi[i];
  }
  if (k3) {
    // byte planes of the eight signed fp16 key entries, index order
    p.klo[0] = p.klo[1] = p.khi[0] = p.khi[1] = 0u;
    for (int e = 0; e < 8; ++e) {
      const uint32_t bits = (k->f16.c16[e / 2] >> (16 * (e % 2))) & 0xFFFFu;
      p.klo[e / 4] |= (bits & 0xFFu) << (8 * (e % 4));
      p.khi[e / 4] |= (bits >> 8) << (8 * (e % 4));
    }
  }
  for (int i = 0; i < 8; ++i) p.kc16[i] = k->f16.c16[i], p.vc16[i] = v->f16.c16[i];
  p.status = k->d_status;
  const bool fixed = k->reserved_smem == (int)RESERVED_SMEM;
  const bool sc = scores_dbg != nullptr;
  const bool v3 = v->fmt == TQ_FMT_TURBO3;
  const dim3 grid(s.grid);
  const cudaError_t e =
      k3 ? (v3 ? launch_t4_variant<true, true>(p, s.heads_per_cta, fixed, sc, grid, st)
               : launch_t4_variant<true, false>(p, s.heads_per_cta, fixed, sc, grid, st))
         : (v3 ? launch_t4_variant<false, true>(p, s.heads_per_cta, fixed, sc, grid, st)
               : launch_t4_variant<false, false>(p, s.heads_per_cta, fixed, sc, grid, st));
  if (e == cudaSuccess && fused) *fused = fuse;
  return e;
}

cudaError_t launch_combine(const tq_ctx *k, const tq_ctx *v, const DecodeShape &s, float *out,
                           const Workspace &ws, cudaStream_t st) {
  (void)k;
  CombineParams p{};
  p.part = ws.partials;
  p.n_heads = s.B * s.Hq;
  p.n_split = s.n_part;
  p.Hq = s.Hq, p.gq = s.gq, p.heads_per_cta = s.heads_per_cta, p.n_hg = s.n_hg;
  p.tiles_per_unit = s.tiles_per_unit, p.vx = s.vx;
  if (!set_schedule(p, s.grid, s.vtotal)) return cudaErrorInvalidValue;
  p.no_main = s.no_main ? 1 : 0;
  p.tail_slot = s.tail_slot;
  const bool vgroup = v->fmt == TQ_FMT_VGROUP2;  // values are not rotated
  p.r = vgroup ? nullptr : v->d_pi;
  p.inv_vscale = 1.0f / (exp2f(P_SHIFT) * (vgroup ? 1.0f : v->f16.alpha));
  p.out = out;
  const size_t smem = (size_t)D * D * 4 + QWARPS * D * 4;
  cudaError_t e = kernel_smem_attr((const void *)k_combine, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_combine, dim3((p.n_heads + QWARPS - 1) / QWARPS), dim3(QWARPS * 32), smem, st, p);
}

cudaError_t launch_combine_prefill(const tq_ctx *v, const PrefillShape &s, float *out,
                                   const Workspace &ws, cudaStream_t st) {
  CombineParams p{};
  p.part = ws.partials;
  p.n_heads = s.B * s.T * s.Hq;
  p.n_split = s.n_part;
  p.Hq = s.Hq, p.gq = s.gq;
  p.tiles_per_unit = s.tiles_per_unit;
  if (!set_schedule(p, s.grid, s.total_tiles)) return cudaErrorInvalidValue;
  p.vx = 0;  // the prefill splits its tiles equally
  p.pf_T = s.T, p.pf_Hkv = s.Hkv, p.pf_qpt = s.qpt, p.pf_n_qt = s.n_qt;
  p.tail_slot = -1;
  p.r = v->d_pi;
  p.inv_vscale = 1.0f / (exp2f(P_SHIFT) * v->f16.alpha);
  p.out = out;
  const size_t smem = (size_t)D * D * 4 + QWARPS * D * 4;
  cudaError_t e = kernel_smem_attr((const void *)k_combine, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_combine, dim3((p.n_heads + QWARPS - 1) / QWARPS), dim3(QWARPS * 32), smem, st, p);
}

}  // namespace tq
