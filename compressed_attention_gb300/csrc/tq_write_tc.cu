// Write path under the dense rotation on the 5th-generation tensor cores: the batched
// rotation Y = X Pi^T ([rows, 128] x [128, 128], "turboquant_plus: how the turbo4 KV
// format came back", section 1 encode chain; "TurboQuant fused Triton kernels deep
// dive", trick 1 for the dense orthogonal Pi) runs as tcgen05 MMAs with the
// accumulator in tensor memory; the canonical fp32 norm n of each row comes from the row
// tile in shared memory, and four threads per row (one per 32-column quarter) finish the
// chain: y = acc / n, nearest centroid through the codebook grid table, packing, scatter.
//
// One persistent CTA per SM takes 128-row tiles blockIdx.x, + gridDim.x, ... (its local
// tiles i = 0, 1, ...) through a warp-specialised pipeline:
//   warp 0      TMA producer: the bf16 rows into a ring of NSTAGE tiles in the 128-byte
//               swizzled K-major layout (two 64-column halves);
//   warp 1      owns the tensor memory (NACC 128-column fp32 accumulators); one thread
//               issues the MMAs of tile i into accumulator i % NACC: Pi split into bf16
//               hi + lo parts, two accumulating products of K = 128, so the rotated
//               coordinates carry about 16 significant bits of Pi against the exact bf16
//               inputs -- enough to keep index decisions identical to the fp64 oracle
//               except within 1e-5 of a decision boundary;
//   warps 2-5   the rows: thread (warp 2 + k, lane) takes row 32 k + lane of the tile --
//               its norm in the canonical order (four-element groups, then the tree
//               p_l + p_{l+16}, + 8, + 4, + 2, + 1), scale / n, its destination slot --
//               into the slot's row data, and (turbo4) stores the norm word;
//   warps 6-21  the epilogue: warp w reads accumulator lanes 32 (w % 4) .. + 31 (the rows
//               of its lane quarter) and columns 32 c .. + 31, c = (w - 6) / 4, and stores
//               its piece of each of the 32 records.
// The row tiles are released once the MMAs and the row warps have read them, so copies and
// products run up to NACC tiles ahead of the epilogue; past the prologue no barrier spans
// more than one warp.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_tc.cuh"

namespace tq {

namespace {

constexpr int NACC = 4;                      // accumulators in tensor memory
constexpr int TC_ROW_WARP0 = 2, TC_EPI_WARP0 = 6;
constexpr int TC_EPI_WARPS = 16;
constexpr int TC_THREADS = 32 * (TC_EPI_WARP0 + TC_EPI_WARPS);
// (22 warps: two of the four schedulers hold six, whose registers come from that
// scheduler's quarter of the register file, 16K: at most 85, so 80 per thread)
constexpr int TC_ROWS = 128;                 // rows per tile (the MMA's M)
constexpr int NSTAGE = 3;                    // row tiles in flight
constexpr uint32_t HALF_BYTES = SW_HALF_BYTES;   // one 64-column half of a bf16 tile
constexpr uint32_t TILE_BYTES = SW_TILE_BYTES;   // 32 KB
static_assert(TC_ROWS == (int)SW_ROWS, "row tiles are the swizzled operand tiles");
constexpr uint32_t TMEM_COLS = 128 * NACC;
static_assert(TMEM_COLS <= 512, "the accumulators fit in tensor memory");
constexpr uint64_t TC_WAIT_NS = 2000000000ull;
constexpr int CELL_COPIES = 16;

// Shared memory: Pi hi (32 KB), Pi lo (32 KB), NSTAGE row tiles (32 KB each), all
// 1024-byte aligned for the 128-byte swizzle; then barriers, the grid table, the row data
// and each epilogue warp's record pieces.
constexpr uint32_t OFF_PIH = 0;
constexpr uint32_t OFF_PIL = TILE_BYTES;
constexpr uint32_t OFF_X = 2 * TILE_BYTES;
constexpr uint32_t OFF_MISC = OFF_X + NSTAGE * TILE_BYTES;
struct TcMisc {
  uint64_t x_full[NSTAGE];      // rows landed (TMA transaction count)
  uint64_t x_empty[NSTAGE];     // rows consumed: the MMAs' commit + one arrival per row warp
  uint64_t acc_full[NACC];      // accumulator written (MMA commit)
  uint64_t row_full[NACC];      // row data of the accumulator's tile written: one arrival per row warp
  uint64_t acc_empty[NACC];     // accumulator and row data read: one arrival per epilogue warp
  uint32_t tmem_addr;
  int abort_flag;
  // grid table in cell coordinates, one copy per half-warp lane (cell t, copy c at 16 t + c,
  // so a warp's lookups of any cells take the minimum two wavefronts): (e[t] * scale +
  // offset, cnt[t] as int bits)
  float2 cell[GRID_CELLS * CELL_COPIES];
  float2 cell0[GRID_CELLS];     // one copy, read from memory
  float nrm[NACC][TC_ROWS];     // row norm
  float su[NACC][TC_ROWS];      // scale / norm (0 for a zero row)
  int64_t slot[NACC][TC_ROWS];  // destination row, -1: not stored
  alignas(16) uint32_t piece[TC_EPI_WARPS][32 * 4];  // each epilogue warp's record pieces (16 bytes per row)
};
static_assert(offsetof(TcMisc, piece) % 16 == 0 && offsetof(TcMisc, cell) % 8 == 0 &&
                  offsetof(TcMisc, slot) % 8 == 0 && OFF_MISC % 16 == 0,
              "vector accesses to the staging are aligned");
constexpr uint32_t SMEM_TC = OFF_MISC + sizeof(TcMisc) + 1024;  // + slack to align the base to 1024
static_assert(SMEM_TC <= 227 * 1024, "one CTA per SM");

struct TcParams {
  const uint16_t *pib;       // Pi hi then lo, bf16 bits [2][128][128] row-major (row j = output j)
  const BucketTable *bt;     // nearest-centroid grid of the codebook
  const int64_t *row_ids;
  uint8_t *dst;
  int64_t n_rows;
  int64_t dst_rows;
  int32_t *status;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane (a warp reads the 32
// lanes of its quarter).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Packed fp32 pairs (two independent round-to-nearest operations, subnormals kept: each
// lane rounds exactly as the scalar operation would).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rr, ra, rb;\n mov.b64 {%0, %1}, rr;\n}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rr, ra, rb;\n mov.b64 {%0, %1}, rr;\n}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rc, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rr, ra, rb, rc;\n mov.b64 {%0, %1}, rr;\n}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

// The four-element partial sums of squares ((x0^2 + x1^2) + (x2^2 + x3^2)) of the two
// groups in a 16-byte chunk (eight bf16: group 0 in words x, y, group 1 in z, w; element
// 2k in the low half of word k), both at once with packed pairs.
__device__ __forceinline__ float2 sq8(uint4 v) {
  const float2 e0 = make_float2(__uint_as_float(v.x << 16), __uint_as_float(v.z << 16));  // x0 of each group
  const float2 e1 = make_float2(__uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.z & 0xFFFF0000u));
  const float2 e2 = make_float2(__uint_as_float(v.y << 16), __uint_as_float(v.w << 16));
  const float2 e3 = make_float2(__uint_as_float(v.y & 0xFFFF0000u), __uint_as_float(v.w & 0xFFFF0000u));
  return add2(add2(mul2(e0, e0), mul2(e1, e1)), add2(mul2(e2, e2), mul2(e3, e3)));
}

template <int FMT>
__global__ void __launch_bounds__(TC_THREADS, 1) k_write_dense_tc(const __grid_constant__ CUtensorMap xmap,
                                                                     const TcParams p) {
  extern __shared__ uint8_t smem_dyn[];
  // 1024-byte aligned base for the swizzled tiles
  uint8_t *smem = smem_dyn + ((1024u - (smem_addr(smem_dyn) & 1023u)) & 1023u);
  TcMisc &ms = *reinterpret_cast<TcMisc *>(smem + OFF_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n_tiles = (p.n_rows + TC_ROWS - 1) / TC_ROWS;
  // local tiles of this CTA: tile = blockIdx.x + i * gridDim.x for i < n_local
  const int n_local = blockIdx.x < n_tiles ? (int)((n_tiles - 1 - blockIdx.x) / gridDim.x) + 1 : 0;
  pdl_trigger();

  if (warp == 1) tmem_alloc(smem_addr(&ms.tmem_addr), TMEM_COLS);
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&ms.x_full[s], 1);
      mbar_init(&ms.x_empty[s], 1 + 4);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&ms.acc_full[b], 1);
      mbar_init(&ms.row_full[b], 4);
      mbar_init(&ms.acc_empty[b], TC_EPI_WARPS);
    }
    ms.abort_flag = 0;
    fence_mbar_init();
    // the first row tiles are requested at once, so they land while Pi is staged (only the
    // source rows need the previous kernel to have finished)
    pdl_wait();
    for (int i = 0; i < NSTAGE && i < n_local; ++i) {
      const int row0 = (int)((blockIdx.x + (int64_t)i * gridDim.x) * TC_ROWS);
      const uint32_t sx = smem_addr(smem + OFF_X) + i * TILE_BYTES;
      mbar_arrive_expect_tx(&ms.x_full[i], TILE_BYTES);
      tma_load_2d(sx, &xmap, &ms.x_full[i], 0, row0);
      tma_load_2d(sx + HALF_BYTES, &xmap, &ms.x_full[i], 64, row0);
    }
  }
  if (tid < GRID_CELLS)  // the grid table: each cell's boundary (mapped like y) and count
    ms.cell0[tid] = make_float2(fmaf(p.bt->e[tid], p.bt->scale, p.bt->offset),
                                __int_as_float(tid < p.bt->n ? (int)p.bt->cnt[tid] : 0));
  {  // Pi hi / lo into the swizzled layout, eight 16-byte loads in flight per thread
    constexpr int N16 = 2 * TC_ROWS * 16;
    for (int i0 = tid; i0 < N16; i0 += 8 * TC_THREADS) {
      uint4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = i0 + k * TC_THREADS;
        if (i < N16) v[k] = reinterpret_cast<const uint4 *>(p.pib)[i];
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = i0 + k * TC_THREADS;
        if (i < N16) {
          const int m = i / (TC_ROWS * 16), rem = i % (TC_ROWS * 16);
          const int row = rem >> 4, chunk = rem & 15;
          *reinterpret_cast<uint4 *>(smem + (m ? OFF_PIL : OFF_PIH) + sw128_offset(row, chunk * 8)) = v[k];
        }
      }
    }
  }
  __syncthreads();
  // the cells' copies, consecutive threads on consecutive entries
  for (int k = tid; k < GRID_CELLS * CELL_COPIES; k += TC_THREADS) ms.cell[k] = ms.cell0[k / CELL_COPIES];
  fence_async_smem();  // generic writes -> tensor-core reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the rows and the cache may be written by the previous kernel
  const uint32_t tmem = ms.tmem_addr;
  const uint32_t sx0 = smem_addr(smem + OFF_X);
  volatile int *abort_flag = &ms.abort_flag;

  if (warp == 0) {
    // ---------------- producer: one thread keeps NSTAGE row tiles in flight
    if (lane == 0) {
      int i = NSTAGE < n_local ? NSTAGE : n_local;  // (the first ones were issued in the prologue)
      for (; i < n_local; ++i) {
        const int s = i % NSTAGE, use = i / NSTAGE;
        if (use > 0 && !mbar_wait_bounded(&ms.x_empty[s], (use - 1) & 1, TC_WAIT_NS)) *abort_flag = 1;
        if (*abort_flag) break;
        const int row0 = (int)((blockIdx.x + (int64_t)i * gridDim.x) * TC_ROWS);
        const uint32_t sx = sx0 + s * TILE_BYTES;
        mbar_arrive_expect_tx(&ms.x_full[s], TILE_BYTES);
        tma_load_2d(sx, &xmap, &ms.x_full[s], 0, row0);
        tma_load_2d(sx + HALF_BYTES, &xmap, &ms.x_full[s], 64, row0);
      }
      // every copy issued has landed before the CTA can leave (after a clean run they were
      // all consumed already)
      for (int j = (i > NSTAGE ? i - NSTAGE : 0); j < i; ++j)
        (void)mbar_wait_bounded(&ms.x_full[j % NSTAGE], (j / NSTAGE) & 1, TC_WAIT_NS);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: Y = X Pi_hi^T + X Pi_lo^T into accumulator i % NACC
    if (lane == 0) {
      const uint32_t spih = smem_addr(smem + OFF_PIH), spil = smem_addr(smem + OFF_PIL);
      int i = 0;
      for (; i < n_local; ++i) {
        const int s = i % NSTAGE, b = i % NACC, use = i / NACC;
        bool ok = mbar_wait_bounded(&ms.x_full[s], (i / NSTAGE) & 1, TC_WAIT_NS);
        if (ok && use > 0) ok = mbar_wait_bounded(&ms.acc_empty[b], (use - 1) & 1, TC_WAIT_NS);
        if (!ok) *abort_flag = 1;
        if (*abort_flag) break;
        tc_fence_after();
        const uint32_t sx = sx0 + s * TILE_BYTES, d = tmem + b * 128;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t sb = part ? spil : spih;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t koff = sw128_kstep(ks);
            umma<IDESC_BF16>(d, sw128_desc(sx + koff), sw128_desc(sb + koff), (part | ks) ? 1u : 0u);
          }
        }
        umma_commit(&ms.acc_full[b]);
        umma_commit(&ms.x_empty[s]);
      }
      // the last MMAs have finished before the tensor memory is released
      if (i > 0) (void)mbar_wait_bounded(&ms.acc_full[(i - 1) % NACC], ((i - 1) / NACC) & 1, TC_WAIT_NS);
    }
  } else if (warp < TC_EPI_WARP0) {
    // ---------------- row warps: row 32 k + lane of every tile
    const int r = 32 * (warp - TC_ROW_WARP0) + lane;
    const float bscale = p.bt->scale;
    for (int i = 0; i < n_local; ++i) {
      const int s = i % NSTAGE, b = i % NACC, use = i / NACC;
      const int64_t row = (blockIdx.x + (int64_t)i * gridDim.x) * TC_ROWS + r;
      // the destination first (its load overlaps the waits)
      const bool live = row < p.n_rows;
      int64_t slot = row;
      if (live && p.row_ids) slot = p.row_ids[row];
      bool ok = mbar_wait_bounded(&ms.x_full[s], (i / NSTAGE) & 1, TC_WAIT_NS);
      if (ok && use > 0) ok = mbar_wait_bounded(&ms.acc_empty[b], (use - 1) & 1, TC_WAIT_NS);
      if (!__all_sync(FULL_MASK, ok)) *abort_flag = 1;
      if (*abort_flag) break;
      // sixteen 16-byte chunks of the row: chunk c holds groups 2 c, 2 c + 1, so pair c
      // of p1 = (p_2c + p_2c+16, p_2c+1 + p_2c+17) -- the tree's first level -- and the
      // levels 8, 4, 2 combine adjacent pairs, in the canonical order
      const uint8_t *xs = smem + OFF_X + s * TILE_BYTES;
      float2 p1[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        p1[c] = add2(sq8(*reinterpret_cast<const uint4 *>(xs + sw128_offset(r, 8 * c))),
                     sq8(*reinterpret_cast<const uint4 *>(xs + sw128_offset(r, 8 * (c + 8)))));
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms.x_empty[s]);  // this warp's reads of the rows are done
#pragma unroll
      for (int h = 4; h >= 1; h >>= 1)
#pragma unroll
        for (int l = 0; l < h; ++l) p1[l] = add2(p1[l], p1[l + h]);
      const float n = __fsqrt_rn(__fadd_rn(p1[0].x, p1[0].y));
      const bool in_range = live && slot >= 0 && slot < p.dst_rows;
      if (live && !in_range) atomicExch(p.status, (int32_t)DEVERR_ROW_OOB);
      ms.nrm[b][r] = n;
      ms.su[b][r] = n == 0.0f ? 0.0f : bscale / n;  // a zero row gives y = 0
      ms.slot[b][r] = in_range ? slot : -1;
      if (FMT == TQ_FMT_TURBO4 && in_range) *reinterpret_cast<float *>(p.dst + slot * 68) = n;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms.row_full[b]);
    }
  } else {
    // ---------------- epilogue: rows 32 qt .. + 31, columns 32 cq .. + 31 of each tile
    const int e = warp - TC_EPI_WARP0, qt = warp & 3, cq = e >> 2;
    const int r = 32 * qt + lane;  // row of the tile (= accumulator lane)
    const float boffset = p.bt->offset;
    const int bn = p.bt->n;
    const float2 *cells = ms.cell + (lane & (CELL_COPIES - 1));
    uint32_t *pc = ms.piece[e];
    for (int i = 0; i < n_local; ++i) {
      const int b = i % NACC, use = i / NACC;
      bool ok = mbar_wait_bounded(&ms.acc_full[b], use & 1, TC_WAIT_NS);
      ok = ok && mbar_wait_bounded(&ms.row_full[b], use & 1, TC_WAIT_NS);
      if (!__all_sync(FULL_MASK, ok)) *abort_flag = 1;
      if (*abort_flag) break;
      tc_fence_after();
      const float su = ms.su[b][r];
      // cell coordinate u = (acc / n) * scale + offset, compared with the boundary in the
      // same coordinates (the decision moves only within rounding of the boundary)
      uint32_t q[4] = {0u, 0u, 0u, 0u};  // turbo4: 32 nibbles; turbo3: 2-bit parts [0..1], high bits [2]
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // columns 32 cq + 16 h .. + 15
        float acc[16];
        tmem_ld16(tmem + ((uint32_t)(32 * qt) << 16) + b * 128 + 32 * cq + 16 * h, acc);
        float uu[16];  // cell coordinates, two per packed FMA
#pragma unroll
        for (int jj = 0; jj < 16; jj += 2) {
          const float2 u2 = fma2(make_float2(acc[jj], acc[jj + 1]), make_float2(su, su), make_float2(boffset, boffset));
          uu[jj] = u2.x, uu[jj + 1] = u2.y;
        }
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int j = 16 * h + jj;
          const float u = uu[jj];
          const uint32_t t = min(__float2uint_rd(u), (uint32_t)(bn - 1));  // NaN, u < 0 -> 0
          const float2 cl = cells[t * CELL_COPIES];
          const uint32_t idx = (uint32_t)__float_as_int(cl.y) + (u > cl.x ? 1u : 0u);
          // (the fields do not overlap: adding places them)
          if (FMT == TQ_FMT_TURBO4) {
            q[j >> 3] += idx << (4 * (j & 7));
          } else {
            q[j >> 4] += (idx & 3u) << (2 * (j & 15));
            q[2] += (idx >> 2) << j;
          }
        }
      }
      const float n = ms.nrm[b][r];
      const int64_t sl_own = ms.slot[b][r];
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms.acc_empty[b]);  // (the row data of the tile are read too)
      // ---- this warp's pieces of its 32 records: staged, then stored by lanes that cover
      // one piece (and, for turbo3, one block) of a record each
      if (FMT == TQ_FMT_TURBO4) {  // words 1 + 4 cq .. + 3
        reinterpret_cast<uint4 *>(pc)[lane] = make_uint4(q[0], q[1], q[2], q[3]);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 4; ++it) {  // rows 8 it + lane / 4, word lane % 4 of the piece
          const int k = 8 * it + (lane >> 2);
          const int64_t sl = __shfl_sync(FULL_MASK, sl_own, k);
          if (sl >= 0) reinterpret_cast<uint32_t *>(p.dst + sl * 68)[1 + 4 * cq + (lane & 3)] = pc[4 * k + (lane & 3)];
        }
      } else {  // block cq: {fp16 norm, qs[8], signs[4]}, 14 bytes at a 2-byte aligned offset
        const uint32_t hn = __half_as_ushort(__float2half_rn(n));
        uint16_t *hp = reinterpret_cast<uint16_t *>(pc);
        hp[7 * lane] = (uint16_t)hn;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          hp[7 * lane + 1 + 2 * k] = (uint16_t)(q[k] & 0xFFFFu);
          hp[7 * lane + 2 + 2 * k] = (uint16_t)(q[k] >> 16);
        }
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 7; ++it) {  // halfword 32 it + lane: halfword j of record k
          const int w = 32 * it + lane, k = w / 7, j = w - 7 * k;
          const int64_t sl = __shfl_sync(FULL_MASK, sl_own, k);
          if (sl >= 0) reinterpret_cast<uint16_t *>(p.dst + sl * 56 + 14 * cq)[j] = hp[w];
        }
      }
      __syncwarp();  // the staging is free for the next tile
    }
  }
  __syncthreads();
  if (tid == 0 && *abort_flag) atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

bool write_tc_eligible(const tq_ctx *ctx, const WriteLaunch &w) {
  if (ctx->p.rotation != TQ_ROT_DENSE || !ctx->d_pib || !ctx->d_bt || ctx->bt.n == 0) return false;
  if (ctx->fmt != TQ_FMT_TURBO4 && ctx->fmt != TQ_FMT_TURBO3) return false;
  if (w.src_dtype != TQ_DTYPE_BF16) return false;
  if ((uintptr_t)w.src % 16 != 0 || (w.stride * 2) % 16 != 0) return false;
  // Small batches (a decode step's few new rows) stay on the CUDA-core kernel, which
  // spreads them over many CTAs; the tensor-core kernel takes whole 128-row tiles.
  if (w.n_rows < 16 * TC_ROWS || w.n_rows > ((int64_t)1 << 31) - TC_ROWS) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_write_tc(const tq_ctx *ctx, const WriteLaunch &w, cudaStream_t st) {
  CUtensorMap map;
  const cuuint64_t dims[2] = {128, (cuuint64_t)w.n_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)w.stride * 2};
  const cuuint32_t box[2] = {64, TC_ROWS};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode_fn()(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w.src), dims, strides,
                                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  TcParams p{};
  p.pib = ctx->d_pib;
  p.bt = ctx->d_bt;
  p.row_ids = w.row_ids;
  p.dst = w.dst;
  p.n_rows = w.n_rows;
  p.dst_rows = w.dst_rows;
  p.status = ctx->d_status;
  const int64_t n_tiles = (w.n_rows + TC_ROWS - 1) / TC_ROWS;
  const int grid = (int)(n_tiles < ctx->num_sms ? n_tiles : ctx->num_sms);  // one persistent CTA per SM
  auto kern = ctx->fmt == TQ_FMT_TURBO4 ? k_write_dense_tc<TQ_FMT_TURBO4> : k_write_dense_tc<TQ_FMT_TURBO3>;
  cudaError_t e = kernel_smem_attr((const void *)kern, (int)SMEM_TC);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(TC_THREADS), SMEM_TC, st, map, p);
}

}  // namespace tq
