// Write path under the dense rotation on the 5th-generation tensor cores: the batched
// rotation Y = X Pi^T ([rows, 128] x [128, 128], "turboquant_plus: how the turbo4 KV
// format came back", section 1 encode chain; "TurboQuant fused Triton kernels deep
// dive", trick 1 for the dense orthogonal Pi) runs as tcgen05 MMAs with the
// accumulator in tensor memory, and two threads per row (one per 64-column half)
// finish the chain: the canonical fp32 norm, y = acc / n, nearest centroid through the
// codebook grid table, packing, scatter.
//
// Per 128-row tile: a TMA load brings the bf16 rows into shared memory in the 128-byte
// swizzled K-major layout (two 64-column halves); the MMA multiplies them by Pi split
// into bf16 hi + lo parts (two accumulating products, K = 128 each), so the rotated
// coordinates carry about 16 significant bits of Pi against the exact bf16 inputs --
// enough to keep index decisions identical to the fp64 oracle except within 1e-5 of a
// decision boundary.  Two CTAs share an SM; each holds Pi (64 KB), one row tile
// (32 KB) and a 128-column fp32 accumulator in tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_tc.cuh"

namespace tq {

namespace {

constexpr int TC_THREADS = 256;        // eight warps: warp w serves rows 32 (w % 4) .. + 31,
                                       // columns 64 (w / 4) .. + 63 of the tile
constexpr int TC_ROWS = 128;           // rows per tile (the MMA's M)
constexpr uint32_t HALF_BYTES = SW_HALF_BYTES;   // one 64-column half of a bf16 tile
constexpr uint32_t TILE_BYTES = SW_TILE_BYTES;   // 32 KB
static_assert(TC_ROWS == (int)SW_ROWS, "row tiles are the swizzled operand tiles");
constexpr uint32_t TMEM_COLS = 128;
constexpr uint64_t TC_WAIT_NS = 2000000000ull;

// Shared memory: Pi hi (32 KB), Pi lo (32 KB), the row tile (32 KB), all 1024-byte
// aligned for the 128-byte swizzle; then barriers, the codebook grid, norms and the
// TMEM address.
constexpr uint32_t OFF_PIH = 0;
constexpr uint32_t OFF_PIL = TILE_BYTES;
constexpr uint32_t OFF_X = 2 * TILE_BYTES;
constexpr uint32_t OFF_MISC = 3 * TILE_BYTES;
struct TcMisc {
  uint64_t x_full;
  uint64_t mma_done;
  uint32_t tmem_addr;
  int abort_flag;
  BucketTable bt;
  float nrm[TC_ROWS];           // row norms
  float upper[TC_ROWS][17];     // group sums 16..31 of each row, handed to the lower half
                                // (padded: rows 17 words apart spread over the banks)
};
constexpr uint32_t SMEM_TC = OFF_MISC + sizeof(TcMisc) + 1024;  // + slack to align the base to 1024

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

template <int FMT>
__global__ void __launch_bounds__(TC_THREADS, 2) k_write_dense_tc(const __grid_constant__ CUtensorMap xmap,
                                                                     const TcParams p) {
  extern __shared__ uint8_t smem_dyn[];
  // 1024-byte aligned base for the swizzled tiles
  uint8_t *smem = smem_dyn + ((1024u - (smem_addr(smem_dyn) & 1023u)) & 1023u);
  TcMisc &ms = *reinterpret_cast<TcMisc *>(smem + OFF_MISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = warp >> 2;               // column half of this thread: 64 * half .. + 63
  const int r = (warp & 3) * 32 + lane;     // row of the tile (= TMEM lane)
  const int64_t n_tiles = (p.n_rows + TC_ROWS - 1) / TC_ROWS;
  pdl_trigger();

  if (warp == 0) tmem_alloc(smem_addr(&ms.tmem_addr), TMEM_COLS);
  if (tid == 0) {
    mbar_init(&ms.x_full, 1);
    mbar_init(&ms.mma_done, 1);
    ms.abort_flag = 0;
    fence_mbar_init();
  }
  {  // the codebook grid, 16-byte pieces
    constexpr int N16 = sizeof(BucketTable) / 16;
    static_assert(sizeof(BucketTable) % 16 == 0, "table copied in 16-byte pieces");
    for (int i = tid; i < N16; i += TC_THREADS)
      reinterpret_cast<uint4 *>(&ms.bt)[i] = reinterpret_cast<const uint4 *>(p.bt)[i];
  }
  {  // Pi hi / lo into the swizzled layout: all 16-byte loads in flight, then the stores
    constexpr int PER = 2 * TC_ROWS * 16 / TC_THREADS;
    uint4 v[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) v[k] = reinterpret_cast<const uint4 *>(p.pib)[tid + k * TC_THREADS];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid + k * TC_THREADS;
      const int m = i / (TC_ROWS * 16), rem = i % (TC_ROWS * 16);
      const int row = rem >> 4, chunk = rem & 15;
      *reinterpret_cast<uint4 *>(smem + (m ? OFF_PIL : OFF_PIH) + sw128_offset(row, chunk * 8)) = v[k];
    }
  }
  fence_async_smem();  // generic writes -> tensor-core reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the rows and the cache may be written by the previous kernel
  const uint32_t tmem = ms.tmem_addr;
  const uint32_t sx = smem_addr(smem + OFF_X);
  const uint32_t spih = smem_addr(smem + OFF_PIH), spil = smem_addr(smem + OFF_PIL);
  const float bscale = ms.bt.scale, boffset = ms.bt.offset;
  const int bn = ms.bt.n;

  if (tid == 0 && blockIdx.x < n_tiles) {
    mbar_arrive_expect_tx(&ms.x_full, TILE_BYTES);
    tma_load_2d(sx, &xmap, &ms.x_full, 0, (int)(blockIdx.x * TC_ROWS));
    tma_load_2d(sx + HALF_BYTES, &xmap, &ms.x_full, 64, (int)(blockIdx.x * TC_ROWS));
  }
  uint32_t phase = 0;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, phase ^= 1u) {
    // ---- wait for the rows, then one thread issues the 16 MMAs
    if (!mbar_wait_bounded(&ms.x_full, phase, TC_WAIT_NS)) ms.abort_flag = 1;
    if (tid == 0 && !ms.abort_flag) {
      tc_fence_after();
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t sb = part ? spil : spih;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t koff = sw128_kstep(ks);
          umma<IDESC_BF16>(tmem, sw128_desc(sx + koff), sw128_desc(sb + koff), (part | ks) ? 1u : 0u);
        }
      }
      umma_commit(&ms.mma_done);
    }
    // ---- canonical fp32 norm: this thread's 16 groups of four, the lower half finishes
    // the tree (p_l + p_{l+16} first, then 8, 4, 2, 1)
    float pl[16];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4 *>(smem + OFF_X + sw128_offset(r, (8 * half + c) * 8));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float x0 = __uint_as_float(w[2 * h] << 16), x1 = __uint_as_float(w[2 * h] & 0xFFFF0000u);
        const float x2 = __uint_as_float(w[2 * h + 1] << 16), x3 = __uint_as_float(w[2 * h + 1] & 0xFFFF0000u);
        pl[2 * c + h] = __fadd_rn(__fadd_rn(__fmul_rn(x0, x0), __fmul_rn(x1, x1)),
                                  __fadd_rn(__fmul_rn(x2, x2), __fmul_rn(x3, x3)));
      }
    }
    if (half) {
#pragma unroll
      for (int l = 0; l < 16; ++l) ms.upper[r][l] = pl[l];
    }
    __syncthreads();
    if (!half) {
#pragma unroll
      for (int l = 0; l < 16; ++l) pl[l] = __fadd_rn(pl[l], ms.upper[r][l]);
#pragma unroll
      for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
        for (int l = 0; l < h; ++l) pl[l] = __fadd_rn(pl[l], pl[l + h]);
      ms.nrm[r] = __fsqrt_rn(pl[0]);
    }
    // ---- accumulator ready; the row tile is no longer needed: prefetch the next one
    if (!mbar_wait_bounded(&ms.mma_done, phase, TC_WAIT_NS)) ms.abort_flag = 1;
    tc_fence_after();
    __syncthreads();
    if (ms.abort_flag) {
      if (tid == 0) {
        atomicExch(p.status, (int32_t)DEVERR_TIMEOUT);
        (void)mbar_wait_bounded(&ms.x_full, phase, TC_WAIT_NS);  // let a late copy land
      }
      break;
    }
    const int64_t next = tile + gridDim.x;
    if (tid == 0 && next < n_tiles) {
      mbar_arrive_expect_tx(&ms.x_full, TILE_BYTES);
      tma_load_2d(sx, &xmap, &ms.x_full, 0, (int)(next * TC_ROWS));
      tma_load_2d(sx + HALF_BYTES, &xmap, &ms.x_full, 64, (int)(next * TC_ROWS));
    }
    // ---- y = acc / n, nearest centroid, pack this thread's 64 columns, store
    const float n = ms.nrm[r];
    const float inv = 1.0f / n;
    const int64_t row = tile * TC_ROWS + r;
    const bool live = row < p.n_rows;
    int64_t slot = row;
    if (live && p.row_ids) slot = p.row_ids[row];
    const bool ok = live && slot >= 0 && slot < p.dst_rows;
    if (live && !ok && half == 0) atomicExch(p.status, (int32_t)DEVERR_ROW_OOB);
    uint32_t q[8];  // turbo4: 64 nibbles; turbo3: 2-bit low parts [0..3], high bits [4..5]
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = 0u;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 64 * half;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      float acc[32];
      tmem_ld32(lane_addr + ch * 32, acc);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float y = (n == 0.0f) ? 0.0f : acc[i] * inv;
        const uint32_t idx = bucket_grid(y, bscale, boffset, bn, ms.bt.cnt, ms.bt.e);
        const int j = ch * 32 + i;  // column within this half
        if (FMT == TQ_FMT_TURBO4) {
          q[j >> 3] |= idx << (4 * (j & 7));
        } else {
          q[j >> 4] |= (idx & 3u) << (2 * (j & 15));
          q[4 + (j >> 5)] |= (idx >> 2) << (j & 31);
        }
      }
    }
    if (ok) {
      if (FMT == TQ_FMT_TURBO4) {
        uint32_t *d = reinterpret_cast<uint32_t *>(p.dst + slot * 68);
        if (half == 0) d[0] = __float_as_uint(n);
#pragma unroll
        for (int i = 0; i < 8; ++i) d[1 + 8 * half + i] = q[i];
      } else {
        // blocks 2 half, 2 half + 1 of {fp16 norm, qs[8], signs[4]}: 28 bytes at a 4-byte
        // aligned offset, assembled as seven words
        const uint32_t hn = __half_as_ushort(__float2half_rn(n));
        uint32_t h16[14];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          h16[7 * c] = hn;
          h16[7 * c + 1] = q[2 * c] & 0xFFFFu;
          h16[7 * c + 2] = q[2 * c] >> 16;
          h16[7 * c + 3] = q[2 * c + 1] & 0xFFFFu;
          h16[7 * c + 4] = q[2 * c + 1] >> 16;
          h16[7 * c + 5] = q[4 + c] & 0xFFFFu;
          h16[7 * c + 6] = q[4 + c] >> 16;
        }
        uint32_t *d = reinterpret_cast<uint32_t *>(p.dst + slot * 56 + 28 * half);
#pragma unroll
        for (int k = 0; k < 7; ++k) d[k] = h16[2 * k] | (h16[2 * k + 1] << 16);
      }
    }
    tc_fence_before();
    __syncthreads();  // accumulator free for the next tile's MMAs
  }
  __syncthreads();
  if (warp == 0) {
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
  const int grid = (int)(n_tiles < 2 * ctx->num_sms ? n_tiles : 2 * ctx->num_sms);
  auto kern = ctx->fmt == TQ_FMT_TURBO4 ? k_write_dense_tc<TQ_FMT_TURBO4> : k_write_dense_tc<TQ_FMT_TURBO3>;
  cudaError_t e = kernel_smem_attr((const void *)kern, (int)SMEM_TC);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(TC_THREADS), SMEM_TC, st, map, p);
}

}  // namespace tq
