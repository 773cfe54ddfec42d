// Fused decode over prod3 keys and vgroup2 values ("TurboQuant fused Triton kernels
// deep dive", tricks 1-3 and "write path and codebook"): every key is scored from its
// 2-bit MSE indices and its 1-bit QJL signs,
//   score = n * ( <q_rot, c[idx]> + gamma * sqrt(pi/2)/d * <S q, sigma> ) * scale,
// with q_rot = Pi q and the sketch S q computed once per query; values are the 2-bit
// group codes, value = code * scale_G + zero_G, never expanded in memory, and not
// rotated, so the combine applies no un-rotation.
//
// Persistent split-K like the turbo4 kernel: one CTA per SM takes a contiguous range
// of 240-key tiles of the (batch, KV head, 8-head group) units; a producer warp
// streams the K (56 B rows) and V (48 B rows) tiles with 1-D bulk copies on a
// four-stage mbarrier ring; fifteen consumer warps take 16 keys each.
//
// MMA orientation (m16n8k16, fp16 operands, fp32 accumulate), per 8-key block:
//   scores  C[16 x 8 keys] = Q[16 x 128] K_hat^T : rows 0-7 hold head g's fp16 hi
//           part, rows 8-15 its lo part, so lane (g, t) ends with head g's exact
//           scores for keys 2t, 2t+1 -- already the layout the PV product takes.
//           The QJL term is a second product with the +-1 signs as the B operand.
//   PV      O^T[128 dims x 8 heads] += codes^T[dims x 16 keys] P_G^T : the codes
//           enter as fp16 subnormal integers (bits = code, value code * 2^-24), the
//           per-key group scale sits in P_G = p * scale_G, split hi + lo into two
//           products with the same codes; each 16-dim m-tile lies inside one group.
// Zero points add sum_t p_t zero_{t,G} per head and group, accumulated in fp32.
#include <math.h>

#include "tq_decode_common.cuh"
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int CW = 15;                 // consumer warps, 16 keys each per tile; with the
                                       // producer 16 warps = 4 per scheduler at 128 registers
constexpr int NTH = (CW + 1) * 32;     // + one producer warp; one CTA per SM
static_assert(16 * CW == PV_TILE, "a tile is 16 keys per consumer warp");
constexpr int NST = 4;                 // pipeline stages
constexpr int K_ROW = 56, V_ROW = 48;
constexpr int K_BUF = PV_TILE * K_ROW + 16;  // start rounded down to 16 B
constexpr int V_BUF = PV_TILE * V_ROW; // V rows start 16-byte aligned

// Key of column c of 8-key block nb.  Chosen so that the packed-word, sign, norm and
// header loads of a warp are free of shared-memory bank conflicts for 56- and 48-byte
// rows (checked exhaustively on the host against the access pattern below).
__constant__ int KEY_ORDER[2][8] = {{7, 15, 3, 11, 13, 5, 1, 9}, {12, 4, 0, 8, 14, 6, 2, 10}};

struct PvParams {
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
  uint32_t kc16[2];   // the four signed fp16 entries alpha * c_k of the 2-bit table
  int32_t *status;
};

struct PvHead {
  float osm[CW][4][D];  // per-warp O of 4 heads (zero terms folded in), for the merge
  uint4 qf[2][8][32];   // the item's q (0) and sketch (1) A fragments: k-step, lane
  float mw[CW][8];
  float lw[CW][8];
  float zw[CW][8][4];
  float mh[8], lh[8];   // an item's per-head max and sum over the warps
  uint64_t full[NST];
  uint64_t empty[NST];
  int abort_flag;
};
// Layout: head, value buffer 0 | MSE table at window LUT_WINDOW | value buffers 1-3,
// key buffers 0-3, sign table.
constexpr uint32_t VBUF0_OFF = (sizeof(PvHead) + 255) & ~255u;
constexpr uint32_t MSE_OFF = LUT_WINDOW - RESERVED_SMEM;        // 256 x 32 slots x 8 B
constexpr uint32_t HIGH_OFF = MSE_OFF + 256 * 32 * 8;
constexpr uint32_t SIGN_OFF = HIGH_OFF + 3 * V_BUF + NST * K_BUF;  // 16 x 32 slots x 8 B
constexpr uint32_t SMEM_PV = SIGN_OFF + 16 * 32 * 8;
static_assert(VBUF0_OFF + V_BUF <= MSE_OFF, "first value buffer below the table");
static_assert(SMEM_PV <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ uint8_t *kbuf(uint8_t *smem, int s) {
  return smem + HIGH_OFF + 3 * V_BUF + s * K_BUF;
}
__device__ __forceinline__ uint8_t *vbuf(uint8_t *smem, int s) {
  return smem + (s == 0 ? VBUF0_OFF : HIGH_OFF + (s - 1) * V_BUF);
}

__device__ __forceinline__ uint2 lds64(const uint8_t *p) { return *reinterpret_cast<const uint2 *>(p); }
__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

// Table entry (two fp16x2 words) at shared-window offset `off` from a table base:
// FIXED puts the base in the load's immediate (the table is at a known window address).
template <bool FIXED, uint32_t WINDOW>
__device__ __forceinline__ void lut2(uint32_t base, uint32_t off, uint32_t &w0, uint32_t &w1) {
  if (FIXED)
    asm("ld.shared.v2.u32 {%0, %1}, [%2+%3];" : "=r"(w0), "=r"(w1) : "r"(off), "n"(WINDOW));
  else
    asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(off + base));
}

template <bool SCORES, bool FIXED>
__global__ void __maxnreg__(128) k_partial_pv(const PvParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  PvHead &sm = *reinterpret_cast<PvHead *>(smem_raw);
  uint32_t *mse_lut = reinterpret_cast<uint32_t *>(smem_raw + MSE_OFF);
  uint32_t *sign_lut = reinterpret_cast<uint32_t *>(smem_raw + SIGN_OFF);
  const int cta = blockIdx.x;
  pdl_trigger();
  if (FIXED && smem_addr(smem_raw) != RESERVED_SMEM) {
    if (threadIdx.x == 0) atomicExch(p.status, (int32_t)DEVERR_LAYOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], CW);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  // MSE table: byte of four 2-bit indices -> (c[i0], c[i1]), (c[i2], c[i3]) as fp16x2,
  // one 8-byte slot per lane.  Sign table: nibble of four QJL bits -> four fp16 +-1.
  for (int piece = threadIdx.x; piece < 256 * 16; piece += NTH) {
    const int byte = piece >> 4, chunk = piece & 15;
    const uint32_t k0 = p.kc16[0], k1 = p.kc16[1];  // (no reference capture: keeps p out of local memory)
    auto c = [k0, k1](int i) { return ((i >> 1 ? k1 : k0) >> (16 * (i & 1))) & 0xFFFFu; };
    const uint32_t w0 = c(byte & 3) | (c((byte >> 2) & 3) << 16);
    const uint32_t w1 = c((byte >> 4) & 3) | (c(byte >> 6) << 16);
    reinterpret_cast<uint4 *>(mse_lut + byte * 64)[chunk] = make_uint4(w0, w1, w0, w1);
  }
  for (int piece = threadIdx.x; piece < 16 * 16; piece += NTH) {
    const int nib = piece >> 4, chunk = piece & 15;
    auto sg = [nib](int i) { return ((nib >> i) & 1) ? 0x3C00u : 0xBC00u; };
    const uint32_t w0 = sg(0) | (sg(1) << 16), w1 = sg(2) | (sg(3) << 16);
    reinterpret_cast<uint4 *>(sign_lut + nib * 64)[chunk] = make_uint4(w0, w1, w0, w1);
  }
  pdl_wait();  // the caches, q and the workspace may be written by the previous kernel
  if (threadIdx.x == 0 && p.seq_lens) {
    for (int b = 0; b < p.B; ++b)
      if (p.seq_lens[b] < 1 || p.seq_lens[b] > p.L) atomicExch(p.status, (int32_t)DEVERR_SEQLEN);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  if (warp == CW) {
    // ---------------- producer
    if (lane == 0) {
      int ctr = 0, tt = cta_first_tile(p, cta);
      Item it;
      bool ok = true;
      while (ok && next_item(p, cta, tt, it)) {
        const int Lb = unit_len(p, it.unit);
        const size_t unit_row0 = (size_t)(it.unit / p.n_hg) * p.L;
        for (int j = it.t0; j < it.t1; ++j) {
          const int kf = j * PV_TILE;
          if (kf >= Lb) break;
          const int nk = min(PV_TILE, Lb - kf);
          const int s = ctr % NST;
          if (ctr >= NST && !mbar_wait_bounded(&sm.empty[s], ((ctr / NST) - 1) & 1, WAIT_LIMIT_NS)) {
            atomicExch(&sm.abort_flag, 1);
            atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
            ok = false;
            break;
          }
          const size_t ks = (unit_row0 + kf) * K_ROW;
          const size_t k0 = ks & ~(size_t)15;
          const size_t k1 = (ks + (size_t)nk * K_ROW + 15) & ~(size_t)15;
          const uint32_t kbytes = (uint32_t)(k1 - k0);
          const uint32_t vbytes = (uint32_t)nk * V_ROW;  // row starts are 16-byte aligned
          mbar_arrive_expect_tx(&sm.full[s], kbytes + vbytes);
          bulk_g2s(kbuf(smem_raw, s), p.kc + k0, kbytes, &sm.full[s]);
          bulk_g2s(vbuf(smem_raw, s), p.vc + (unit_row0 + kf) * V_ROW, vbytes, &sm.full[s]);
          ++ctr;
        }
      }
      if (!ok || sm.abort_flag) {
        for (int c = (ctr > NST ? ctr - NST : 0); c < ctr; ++c)
          (void)mbar_wait_bounded(&sm.full[c % NST], (c / NST) & 1, WAIT_LIMIT_NS);
      }
    }
    return;
  }

  // ---------------- consumers
  const uint32_t mse_base = smem_addr(mse_lut), sign_base = smem_addr(sign_lut);
  constexpr uint32_t SIGN_WINDOW = RESERVED_SMEM + SIGN_OFF;
  const uint32_t laneword = 8u * lane;
  const int kb = warp * 16;
  const int kr0 = KEY_ORDER[0][g], kr1 = KEY_ORDER[1][g];  // B-operand keys (column g)
  int ks[4];                                               // this lane's softmax / PV keys
  ks[0] = KEY_ORDER[0][2 * t], ks[1] = KEY_ORDER[0][2 * t + 1];
  ks[2] = KEY_ORDER[1][2 * t], ks[3] = KEY_ORDER[1][2 * t + 1];
  const uint32_t code_sel = (uint32_t)(g & 3) | ((4u + (g & 3)) << 8);
  const int code_word = 4 * (g >> 2);  // byte offset of word (g >> 2) inside a group

  int ctr = 0, tt = cta_first_tile(p, cta);
  Item it;
  bool aborted = false;
  while (!aborted && next_item(p, cta, tt, it)) {
    const int Lb = unit_len(p, it.unit);
    const int hg = it.unit % p.n_hg;
    const int bk = it.unit / p.n_hg;
    const int b = bk / p.Hkv, kvh = bk % p.Hkv;
    const int G = min(8, p.gq - hg * 8);
    const int head0 = kvh * p.gq + hg * 8;
    const size_t unit_row0 = (size_t)bk * p.L;

    // q and the sketch S q as A operands: rows g / g+8 = fp16 hi / lo of head g; k-step
    // s covers dims 32t + 4s .. 32t + 4s + 3 in lane t.  The fragments of the item are
    // written to shared memory once by all consumer warps (the previous item's merge ended
    // with their barrier) and read at each k-step.
    for (int i = threadIdx.x; i < 2 * 8 * 32; i += CW * 32) {
      const int which = i >> 8, st = (i >> 5) & 7, ln = i & 31;
      const int fg = ln >> 2, ft = ln & 3, v = st >> 1, h = st & 1;
      uint4 f = make_uint4(0u, 0u, 0u, 0u);
      if (fg < G) {
        const uint4 *qw = reinterpret_cast<const uint4 *>(p.qhl + (size_t)(b * p.Hq + head0 + fg) * 256);
        const uint4 hi = qw[32 * which + 4 * ft + v], lo = qw[32 * which + 16 + 4 * ft + v];
        const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w}, lw[4] = {lo.x, lo.y, lo.z, lo.w};
        f = make_uint4(hw[2 * h], lw[2 * h], hw[2 * h + 1], lw[2 * h + 1]);
      }
      sm.qf[which][st][ln] = f;
    }
    float qsm = 0.f, qsq = 0.f;
    if (g < G) {
      qsm = p.qsc[2 * (b * p.Hq + head0 + g)];
      qsq = p.qsc[2 * (b * p.Hq + head0 + g) + 1];
    }
    named_sync1<CW * 32>();
    float O[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) O[mt][0] = O[mt][1] = O[mt][2] = O[mt][3] = 0.f;
    float M = -INFINITY, lsum = 0.f, zt[4] = {0.f, 0.f, 0.f, 0.f};

    for (int j = it.t0; j < it.t1; ++j) {
      const int kf = j * PV_TILE;
      if (kf >= Lb) break;
      const int s = ctr % NST;
      if (!mbar_wait_bounded(&sm.full[s], (ctr / NST) & 1, WAIT_LIMIT_NS)) {
        if (lane == 0) {
          atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
          atomicExch(&sm.abort_flag, 1);
        }
        aborted = true;
        break;
      }
      if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) {
        aborted = true;
        break;
      }
      const int nk = min(PV_TILE, Lb - kf);
      const size_t kstart = (unit_row0 + kf) * K_ROW;
      const uint8_t *Ks = kbuf(smem_raw, s) + (kstart & 15) + kb * K_ROW;
      const uint8_t *Vs = vbuf(smem_raw, s) + kb * V_ROW;
      const int nkb = nk - kb;
      if (nkb > 0) {
        // ---- scores of two 8-key blocks: MSE and QJL products
        // even and odd k-steps accumulate separately (two chains of four dependent MMAs
        // each instead of one of eight), summed once after the loop
        float cm[2][2][4], cq[2][2][4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int h = 0; h < 2; ++h) cm[h][0][e] = cm[h][1][e] = cq[h][0][e] = cq[h][1][e] = 0.f;
        const uint2 m0 = lds64(Ks + kr0 * K_ROW + 8 + 8 * t), m1 = lds64(Ks + kr1 * K_ROW + 8 + 8 * t);
        const uint32_t sw0 = lds32(Ks + kr0 * K_ROW + 40 + 4 * t), sw1 = lds32(Ks + kr1 * K_ROW + 40 + 4 * t);
        const uint32_t ev0 = sw0 & 0x0F0F0F0Fu, od0 = (sw0 >> 4) & 0x0F0F0F0Fu;
        const uint32_t ev1 = sw1 & 0x0F0F0F0Fu, od1 = (sw1 >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const uint32_t mw0 = st < 4 ? m0.x : m0.y, mw1 = st < 4 ? m1.x : m1.y;
          const uint32_t nw0 = (st & 1) ? od0 : ev0, nw1 = (st & 1) ? od1 : ev1;
          uint32_t b00, b01, b10, b11, s00, s01, s10, s11;
          // table offsets: byte st & 3 of the MSE word, nibble-byte st >> 1 of the sign word
          const uint32_t selm = 0x1100u | ((4u + (st & 3)) << 4), seln = 0x1100u | ((4u + (st >> 1)) << 4);
          const uint32_t om0 = prmt(laneword, mw0, selm), om1 = prmt(laneword, mw1, selm);
          const uint32_t on0 = prmt(laneword, nw0, seln), on1 = prmt(laneword, nw1, seln);
          lut2<FIXED, LUT_WINDOW>(mse_base, om0, b00, b01);
          lut2<FIXED, LUT_WINDOW>(mse_base, om1, b10, b11);
          lut2<FIXED, SIGN_WINDOW>(sign_base, on0, s00, s01);
          lut2<FIXED, SIGN_WINDOW>(sign_base, on1, s10, s11);
          const uint4 fa = sm.qf[0][st][lane], fq = sm.qf[1][st][lane];
          const uint32_t qa[4] = {fa.x, fa.y, fa.z, fa.w}, qq[4] = {fq.x, fq.y, fq.z, fq.w};
          mma_f16(cm[st & 1][0], qa, b00, b01);
          mma_f16(cm[st & 1][1], qa, b10, b11);
          mma_f16(cq[st & 1][0], qq, s00, s01);
          mma_f16(cq[st & 1][1], qq, s10, s11);
        }
        // ---- online softmax for head g over keys ks[0..3]
        float sc[4], u[4], tn[4];
        uint4 hv[4];  // value headers: word G = (fp16 scale_G, fp16 zero_G)
        bool ok[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kr = ks[i];
          ok[i] = kr < nkb;
          const float2 ng = *reinterpret_cast<const float2 *>(Ks + kr * K_ROW);
          hv[i] = *reinterpret_cast<const uint4 *>(Vs + kr * V_ROW + 32);
          if (!ok[i]) hv[i] = make_uint4(0u, 0u, 0u, 0u);
          // nu = fp16 exponent of the largest scale minus 14, so scale * 2^-nu < 1 for every
          // group (scales are >= 0, so their fp16 bit patterns order like their values)
          const uint32_t mb = __vmaxu2(__vmaxu2(hv[i].x, hv[i].y), __vmaxu2(hv[i].z, hv[i].w));
          const int nu = (int)((mb >> 10) & 0x1Fu) - 14;
          tn[i] = __uint_as_float((uint32_t)(127 - nu) << 23);
          const int nb = i >> 1, e = i & 1;
          const float mse = (cm[0][nb][e] + cm[0][nb][2 + e]) + (cm[1][nb][e] + cm[1][nb][2 + e]);
          const float qjl = (cq[0][nb][e] + cq[0][nb][2 + e]) + (cq[1][nb][e] + cq[1][nb][2 + e]);
          sc[i] = ok[i] ? ng.x * fmaf(ng.y * qsq, qjl, qsm * mse) : -INFINITY;
          u[i] = sc[i] + (float)nu;
          if (SCORES && ok[i] && g < G)
            p.scores[(size_t)(b * p.Hq + head0 + g) * p.L + kf + kb + kr] = sc[i] * LN2;
        }
        float bm = fmaxf(fmaxf(u[0], u[1]), fmaxf(u[2], u[3]));
        bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 2));
        const bool need = bm > M + RESCALE_SLACK;  // also taken while M is -inf
        if (__any_sync(FULL_MASK, need)) {
          const float alpha = need ? exp2_approx(M - bm) : 1.f;
          if (need) M = bm;
          lsum *= alpha;
#pragma unroll
          for (int G4 = 0; G4 < 4; ++G4) zt[G4] *= alpha;
          const float aa = __shfl_sync(FULL_MASK, alpha, 8 * t), ab = __shfl_sync(FULL_MASK, alpha, 8 * t + 4);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) O[mt][0] *= aa, O[mt][1] *= ab, O[mt][2] *= aa, O[mt][3] *= ab;
        }
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float pp[4], pw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          lsum += exp2_approx(sc[i] - Mu);
          pp[i] = exp2_approx(u[i] - Mu + P_SHIFT);  // 2^(s - M + P) * 2^nu
          pw[i] = pp[i] * tn[i];                      // 2^(s - M + P)
        }
        // ---- PV per group: codes as the A operand, p * scale_G (hi + lo) as B; the
        // zero points accumulate in fp32.
#pragma unroll
        for (int G4 = 0; G4 < 4; ++G4) {
          float sg[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t w = G4 == 0 ? hv[i].x : G4 == 1 ? hv[i].y : G4 == 2 ? hv[i].z : hv[i].w;
            const float2 sz = __half22float2(*reinterpret_cast<const __half2 *>(&w));
              sg[i] = pw[i] * sz.x;  // 2^(s - M + P) * scale_G <= p' (scale * 2^-nu < 1)
            zt[G4] = fmaf(pw[i], sz.y, zt[G4]);
          }
          uint32_t b0h, b0l, b1h, b1l;
          split_half2(sg[0], sg[1], b0h, b0l);
          split_half2(sg[2], sg[3], b1h, b1l);
          const int wo = 8 * G4 + code_word;
          const uint32_t wa = lds32(Vs + ks[0] * V_ROW + wo), wb = lds32(Vs + ks[1] * V_ROW + wo);
          const uint32_t wc = lds32(Vs + ks[2] * V_ROW + wo), wd = lds32(Vs + ks[3] * V_ROW + wo);
          const uint32_t zab = prmt(wa, wb, code_sel), zcd = prmt(wc, wd, code_sel);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t a[4] = {(zab >> (4 * h)) & 0x00030003u, (zab >> (4 * h + 2)) & 0x00030003u,
                                   (zcd >> (4 * h)) & 0x00030003u, (zcd >> (4 * h + 2)) & 0x00030003u};
            mma_f16(O[2 * G4 + h], a, b0h, b1h);
            mma_f16(O[2 * G4 + h], a, b0l, b1l);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
      ++ctr;
    }
    if (aborted || *reinterpret_cast<volatile int *>(&sm.abort_flag)) break;
    lsum += __shfl_xor_sync(FULL_MASK, lsum, 1);
    lsum += __shfl_xor_sync(FULL_MASK, lsum, 2);
#pragma unroll
    for (int G4 = 0; G4 < 4; ++G4) {
      zt[G4] += __shfl_xor_sync(FULL_MASK, zt[G4], 1);
      zt[G4] += __shfl_xor_sync(FULL_MASK, zt[G4], 2);
    }

    // ---- merge the consumer warps' states of this item and write its partial: the
    // per-head max and sum over the warps by eight lanes of warp 0, then the accumulators
    // in two passes of four heads through osm
    if (t == 0) {
      sm.mw[warp][g] = M;
      sm.lw[warp][g] = lsum;
#pragma unroll
      for (int G4 = 0; G4 < 4; ++G4) sm.zw[warp][g][G4] = zt[G4];
    }
    named_sync1<CW * 32>();
    if (warp == 0 && lane < 8) {
      float ms = -INFINITY;
      for (int w = 0; w < CW; ++w) ms = fmaxf(ms, sm.mw[w][lane]);
      float v = 0.f;
      if (ms != -INFINITY)
        for (int w = 0; w < CW; ++w)
          if (sm.mw[w][lane] != -INFINITY) v += sm.lw[w][lane] * exp2_approx(sm.mw[w][lane] - ms);
      sm.mh[lane] = ms, sm.lh[lane] = v;
    }
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      if ((t >> 1) == pass) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hh = 2 * t + e;  // head of accumulator columns c0/c2 (e = 0), c1/c3 (e = 1)
          float ms = -INFINITY;
          for (int w = 0; w < CW; ++w) ms = fmaxf(ms, sm.mw[w][hh]);
          const float mine = sm.mw[warp][hh];
          const float fac = (mine == -INFINITY) ? 0.f : exp2_approx(mine - ms);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const int G4 = mt >> 1;
            const float z = sm.zw[warp][hh][G4];
            const int d0 = 32 * G4 + 4 * g + 2 * (mt & 1);
            sm.osm[warp][hh - 4 * pass][d0] = fmaf(O[mt][e], 16777216.f, z) * fac;
            sm.osm[warp][hh - 4 * pass][d0 + 1] = fmaf(O[mt][2 + e], 16777216.f, z) * fac;
          }
        }
      }
      named_sync1<CW * 32>();
      const int Gp = min(4, G - 4 * pass);
      for (int idx = threadIdx.x; idx < Gp * D; idx += CW * 32) {
        const int h4 = idx / D, jd = idx % D, hh = 4 * pass + h4;
        const float ms = sm.mh[hh];
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < CW; ++w) acc += sm.osm[w][h4][jd];
        float *dst = p.part + ((size_t)(b * p.Hq + head0 + hh) * p.n_part + it.slot) * PARTIAL_FLOATS;
        dst[6 + jd] = (ms == -INFINITY) ? 0.f : acc;
        if (jd < 6) dst[jd] = jd == 0 ? ms : (jd == 1 ? sm.lh[hh] : 0.f);
      }
      named_sync1<CW * 32>();
    }
  }
}

template <bool SC, bool FIXED>
cudaError_t launch_pv(const PvParams &p, dim3 grid, cudaStream_t st) {
  auto kern = k_partial_pv<SC, FIXED>;
  cudaError_t e = kernel_smem_attr((const void *)kern, (int)SMEM_PV, true);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(NTH), SMEM_PV, st, p);
}

}  // namespace

cudaError_t launch_partial_pv(const tq_ctx *k, const tq_ctx *v, const uint8_t *kc,
                              const uint8_t *vc, const int32_t *seq_lens, const DecodeShape &s,
                              float *scores_dbg, const Workspace &ws, cudaStream_t st) {
  (void)v;
  PvParams p{};
  p.kc = kc, p.vc = vc, p.seq_lens = seq_lens;
  p.B = s.B, p.Hq = s.Hq, p.Hkv = s.Hkv, p.L = s.L, p.gq = s.gq, p.n_hg = s.n_hg;
  p.tiles_per_unit = s.tiles_per_unit, p.vx = s.vx;
  if (!set_schedule(p, s.grid, s.vtotal)) return cudaErrorInvalidValue;
  p.total_tiles = s.total_tiles, p.n_part = s.n_part;
  p.qhl = ws.qhl, p.qsc = ws.qsc, p.part = ws.partials, p.scores = scores_dbg;
  p.kc16[0] = k->f16.c16[0], p.kc16[1] = k->f16.c16[1];
  p.status = k->d_status;
  dim3 grid(s.grid);
  const bool fixed = k->reserved_smem == (int)RESERVED_SMEM;
  if (fixed) return scores_dbg ? launch_pv<true, true>(p, grid, st) : launch_pv<false, true>(p, grid, st);
  return scores_dbg ? launch_pv<true, false>(p, grid, st) : launch_pv<false, false>(p, grid, st);
}

}  // namespace tq
