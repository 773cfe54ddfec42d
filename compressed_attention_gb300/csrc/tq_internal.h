// Internal declarations shared by the host library and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

constexpr int D = 128;
// Head dimension 256 (turbo4): a row is two consecutive 68-byte turbo4 blocks.
constexpr int D256 = 256;
constexpr int ROW256 = 136;
constexpr int ACC256 = 8;                 // a d = 256 partial: max, sum, 6 spare, acc[256]
constexpr int PARTIAL256 = ACC256 + D256;

// Device status codes (see tq_ctx_device_status in tq.h).
enum DevErr : int32_t { DEVERR_ROW_OOB = 1, DEVERR_SEQLEN = 2, DEVERR_TIMEOUT = 3, DEVERR_LAYOUT = 4 };

// Stored codebook: K fp32 centroids and K-1 fp32 decision boundaries.
struct Codebook {
  int bits = 0;
  int K = 0;
  float c[16] = {};
  float b[15] = {};
};

// fp16 operand table of a symmetric codebook for the tensor-core decode.
// Magnitude m (0 = largest) of the scaled centroid alpha*|c_m| as fp16; byte
// planes split for prmt lookups: lo[] holds the low bytes of entries 0..7, hi[]
// the high bytes.  alpha is chosen so the fp16 rounding error of all entries
// is smallest (it is divided out again after the products).
struct F16Table {
  uint32_t lo[2] = {0, 0};
  uint32_t hi[2] = {0, 0};
  uint32_t c16[8] = {};  // the K signed fp16 entries (alpha * c_k), two per word, index order
  float alpha = 1.0f;
  float max_rel_err = 0.0f;
};

// Nearest-centroid decision through a uniform grid over the decision boundaries.
// Cells are 2/5 of the smallest boundary gap wide, so a cell widened by delta (5% of a
// cell) on each side holds at most one boundary: cell t stores cnt[t] = #{k : b_k <
// left edge - delta} and that boundary (+inf when none), and idx(y) = #{k : y > b_k} =
// cnt[t] + [y > e[t]] for every y whose computed cell t = clamp(floor(y * scale +
// offset), 0, n - 1) -- the fp32 cell computation errs by far less than delta.
// n == 0: the table is unusable (binary search instead).
constexpr int GRID_CELLS = 160;
struct alignas(16) BucketTable {
  float scale = 0.f, offset = 0.f;
  int n = 0, pad = 0;
  uint8_t cnt[GRID_CELLS] = {};
  float e[GRID_CELLS] = {};
};

}  // namespace tq

struct tq_ctx {
  tq_params p{};
  int device = 0;
  int num_sms = 0;
  int reserved_smem = 0;  // shared-window bytes reserved before dynamic shared memory
  int fmt = 0;
  tq::Codebook cb{};
  tq::F16Table f16{};
  int d = 128;                         // head dimension: 128, or 256 (turbo4)
  uint32_t wht_neg[8] = {};             // bit j set: WHT sign j is -1
  float *d_pi = nullptr;                // rotation R (dense Pi or the WHT matrix), fp32 row-major
  float *d_pit = nullptr;               // R^T, fp32 row-major
  float *d_S = nullptr;                 // QJL matrix S, fp32 [128][128] row-major
  float *d_St = nullptr;                // S^T, fp32 row-major
  uint16_t *d_pib = nullptr;            // dense R as bf16 hi then lo, [2][128][128] (tensor-core write)
  tq::BucketTable bt{};                 // nearest-centroid grid of the codebook (host copy)
  tq::BucketTable *d_bt = nullptr;      // the same on the device
  int32_t *d_status = nullptr;          // device status word
  float qjl_factor = 1.0f;              // PROD3 reads: 1 (unbiased) or 2/pi (shrunk QJL term)
};

namespace tq {

// Launch with programmatic stream serialization: the kernel may begin its prologue
// while the previous kernel on the stream finishes (it waits with pdl_wait before
// touching anything that kernel may write).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ---- host helpers (tq_host.cpp) ----
bool make_codebook_f64(int bits, int d, int kind, double *c);
void store_codebook(const double *c64, int K, float *c32, float *b32);
void splitmix64_fill(uint64_t seed, uint64_t *out, size_t n);
void gaussian_fill(uint64_t seed, double *out, size_t n);
bool dense_rotation_f64(uint64_t seed, int d, double *pi);
F16Table make_f16_table(const float *c32, int K);
BucketTable make_bucket_table(const float *b, int nb);
void set_error(const char *fmt, ...);
// TQ_OK when `device` is the calling thread's current device; else TQ_ERR_INVALID_ARG
// (or TQ_ERR_CUDA when the current device cannot be read), with the reason recorded.
// Every call that launches work checks its contexts' device this way: their tables and
// status word live in that device's memory, and the kernels run on the current one.
tq_status check_current_device(int device, const char *who);
// Raises a kernel's dynamic shared-memory limit to `bytes` (and, with max_shared, asks for
// the largest shared-memory carveout) once per (kernel, device, setting): the attribute
// stays with the function on that device, so later launches skip the driver calls.
cudaError_t kernel_smem_attr(const void *func, int bytes, bool max_shared = false);
// Resident CTAs per SM of a kernel at `threads` threads and `smem` bytes of dynamic shared
// memory, asked of the runtime once per (kernel, device, launch shape).
cudaError_t kernel_occupancy(const void *func, int threads, size_t smem, int *blocks);

// ---- kernel launchers ----
struct WriteLaunch {
  const void *src;
  int src_dtype;
  int64_t n_rows;
  int64_t stride;
  const int64_t *row_ids;
  uint8_t *dst;
  int64_t dst_rows;
};
cudaError_t launch_write(const tq_ctx *ctx, const WriteLaunch &w, cudaStream_t st);
// The decode step's front in one launch (tq_decode_step): both small-batch dense writes and
// the q preparation; eligible for dense-rotation turbo4 / turbo3 caches and at most 256 rows.
struct QprepParams;
bool step_front_eligible(const tq_ctx *k, const tq_ctx *v, const WriteLaunch &wk, const WriteLaunch &wv);
cudaError_t launch_step_front(const tq_ctx *k, const tq_ctx *v, const WriteLaunch &wk, const WriteLaunch &wv,
                              const QprepParams &q, cudaStream_t st);
// prod3 keys, vgroup2 values: the same one-launch front (K rows by CTA, V rows by warp, q with its sketch)
bool step_front_pv_eligible(const tq_ctx *k, const tq_ctx *v, const WriteLaunch &wk, const WriteLaunch &wv);
cudaError_t launch_step_front_pv(const tq_ctx *k, const tq_ctx *v, const WriteLaunch &wk, const WriteLaunch &wv,
                              const QprepParams &q, cudaStream_t st);
bool write_tc_eligible(const tq_ctx *ctx, const WriteLaunch &w);
cudaError_t launch_write_tc(const tq_ctx *ctx, const WriteLaunch &w, cudaStream_t st);

cudaError_t launch_dequantize(const tq_ctx *ctx, const uint8_t *cache, int64_t n_rows,
                              int unrotate, float *dst, cudaStream_t st);

constexpr int T4_TILE = 240;  // keys per tile of the turbo4 decode
constexpr int PV_TILE = 240;  // keys per tile of the prod3-key / vgroup2-value decode
// Fixed cost of one more work item in a CTA's range (the consumer warps' merge, the
// partial's write, the next unit's q), in tiles of the kernel's own streaming time.
constexpr int T4_ITEM_TILES = 4;
constexpr int T3_ITEM_TILES = 3;  // turbo3 keys: longer tiles
constexpr int PV_ITEM_TILES = 2;

struct DecodeShape {
  int B, Hq, Hkv, L;
  int tile;     // keys per tile (T4_TILE or PV_TILE)
  bool pv;      // prod3 keys with vgroup2 values
  int gq;       // q-heads per KV head
  int heads_per_cta;  // q-heads one CTA serves (4 or 8)
  int n_hg;     // head groups per KV head
  int tiles_per_unit;  // key tiles of one (batch, KV head, head group) unit
  int total_tiles;     // over all units, laid end to end
  int vtotal;          // virtual tiles: each unit counts vx tiles of item cost ahead of its own
  int tiles_per_cta;   // longest CTA range, in virtual tiles (CTA c takes virtual tiles
                       // [c * vtotal / grid, (c + 1) * vtotal / grid), rounded down)
  int vx;
  int grid;            // persistent CTAs (at most one per SM)
  int n_part;          // partial slots per head
  int tail_slot = -1;  // slot of an exact-tail partial (the store's ring), or -1
  bool no_main = false;  // no split-K partials: every key is in the exact tail
};
struct Workspace {
  uint32_t *qhl;     // [B*Hq][2 operands][128 fp16]: hi then lo, per operand (q_rot, sketch)
  float *qsc;        // [B*Hq][2] power-of-two scales of the two operands
  float *partials;   // [B*Hq][n_split][PARTIAL_FLOATS]
  int32_t *unit_done;  // [units] CTAs that wrote their partial of a unit (fused combine);
                       // zeroed by the q preparation
  int n_units;
  size_t bytes;
};
constexpr int PARTIAL_FLOATS = 2 + 4 + D;  // max, sum, 4 group zero-terms, acc[128]

// Arguments of the q preparation (tq_qprep.cuh).
struct QprepParams {
  const void *q;
  int q_dtype;
  int n_q;            // B * Hq
  const float *r;     // R, fp32 [128][128] row-major
  const float *s;     // S for the QJL sketch (prod3 keys), row-major, or null
  float mul;          // log2(e) * scale / alpha_K
  float mul_sk;       // log2(e) * scale * sqrt(pi/2) / d (sketch)
  uint32_t *qhl;
  float *qsc;
  int32_t *unit_done;  // zeroed there for the fused combine of the next split-K launch
  int n_units;
};

bool decode_shape(const tq_ctx *k, const tq_ctx *v, int B, int Hq, int Hkv, int L,
                  DecodeShape *s);
bool decode_pair_supported(const tq_ctx *k, const tq_ctx *v);  // a decode kernel exists
Workspace carve_workspace(const DecodeShape &s, void *base);

// Head dimension 256 (tq_d256.cu): turbo4 keys and values only.
struct D256Shape {
  int B, Hq, Hkv, L, gq, n_hg;  // units: (batch, KV head, group of up to 4 q-heads)
  int n_split, chunk;          // splits per unit, keys per split (a multiple of 16)
  int units;
};
bool d256_shape(const tq_ctx *k, int B, int Hq, int Hkv, int L, D256Shape *s);
size_t d256_workspace(const D256Shape &s, void *base, Workspace *w);  // returns the bytes
cudaError_t launch_write_d256(const tq_ctx *ctx, const WriteLaunch &w, cudaStream_t st);
cudaError_t launch_dequant_d256(const tq_ctx *ctx, const uint8_t *cache, int64_t n_rows, int unrotate,
                                float *dst, cudaStream_t st);
cudaError_t launch_prepare_q256(const tq_ctx *k, const void *q, int q_dtype, const D256Shape &s, float scale,
                                const Workspace &w, cudaStream_t st);
cudaError_t launch_partial_d256(const tq_ctx *k, const tq_ctx *v, const uint8_t *kc, const uint8_t *vc,
                                const int32_t *seq_lens, const D256Shape &s, const Workspace &w, cudaStream_t st);
cudaError_t launch_combine_d256(const tq_ctx *v, const D256Shape &s, float *out, const Workspace &w,
                                cudaStream_t st);

QprepParams make_qprep_params(const tq_ctx *k, const void *q, int q_dtype, const DecodeShape &s,
                              float scale, const Workspace &ws);
cudaError_t launch_prepare_q(const tq_ctx *k, const void *q, int q_dtype, const DecodeShape &s,
                             float scale, const Workspace &ws, cudaStream_t st);
bool partial_fuses_combine(const DecodeShape &s);  // tq_decode_attention skips the combine
// out != null asks for the combine fused into the split-K kernel (the CTA that completes a
// unit merges it and writes the outputs); *fused tells whether it was (else launch_combine).
cudaError_t launch_partial(const tq_ctx *k, const tq_ctx *v, const uint8_t *kc,
                           const uint8_t *vc, const int32_t *seq_lens, const DecodeShape &s,
                           float *scores_dbg, const Workspace &ws, cudaStream_t st,
                           bool withhold_first_tile = false, float *out = nullptr,
                           bool *fused = nullptr);
cudaError_t launch_partial_pv(const tq_ctx *k, const tq_ctx *v, const uint8_t *kc,
                              const uint8_t *vc, const int32_t *seq_lens, const DecodeShape &s,
                              float *scores_dbg, const Workspace &ws, cudaStream_t st);
cudaError_t launch_combine(const tq_ctx *k, const tq_ctx *v, const DecodeShape &s, float *out,
                           const Workspace &ws, cudaStream_t st);

// Chunked prefill over the compressed cache: T queries per sequence at positions
// q_start[b] .. q_start[b] + T - 1, units (batch, KV head, tile of qpt queries x gq heads).
constexpr int PF_TILE = 128;  // keys per tile of the prefill
struct PrefillShape {
  int B, T, Hq, Hkv, L;
  int gq;              // q-heads per KV head (a divisor of 128)
  int qpt;             // queries per unit: 128 / gq rows
  int n_qt;            // query tiles per (batch, KV head)
  int tiles_per_unit;  // key tiles of one unit (all of L; tiles past a unit's last
                       // visible key cost no work)
  int total_tiles, tiles_per_cta, grid, n_part;  // tiles_per_cta: the longest CTA range
  DecodeShape q;       // the B*T queries as a decode batch: q preparation and workspace
};
bool prefill_shape(const tq_ctx *k, int B, int T, int Hq, int Hkv, int L, PrefillShape *s);
cudaError_t launch_prefill(const tq_ctx *k, const tq_ctx *v, const uint8_t *kc, const uint8_t *vc,
                           const int32_t *q_start, const PrefillShape &s, const Workspace &ws,
                           cudaStream_t st);
cudaError_t launch_combine_prefill(const tq_ctx *v, const PrefillShape &s, float *out,
                                   const Workspace &ws, cudaStream_t st);

}  // namespace tq
