/*
 * tq.h -- C ABI of the GB300 compressed-KV library (TurboQuant-style KV-cache
 * compression: write path = quantize / SET_ROWS, read path = fused decode
 * attention over the packed cache).
 *
 * Sources for the operations (page title, section):
 *   [turbo4 post-mortem]  "turboquant_plus: how the turbo4 KV format came back",
 *                         sections 1 (encode chain: norm -> normalise -> random
 *                         rotation -> nearest centroid), 2 (SET_ROWS bugs),
 *                         4 (dequant by direct extraction), 5 (16-centroid
 *                         turbo4, nibble packing), 7 (68-byte block), 9, 10.
 *   [Triton deep dive]    "TurboQuant fused Triton kernels deep dive", tricks
 *                         1-3 (rotate q once, QJL query sketch once, single-pass
 *                         online softmax with in-register value dequant) and
 *                         "write path and codebook" (Lloyd-Max codebook, 2-bit
 *                         group value quantization).
 *
 * Conventions common to every call
 *   - Head dimension d = 128 for every format, and d = 256 for TURBO4 ([turbo4
 *     post-mortem] section 9, per-head-dimension codebooks): a 256-element row is
 *     rotated as a whole, quantized with the codebook of N(0, 1/256), and stored as
 *     two consecutive 68-byte TURBO4 blocks (elements 128c .. 128c+127 in block c,
 *     the row's norm in both), each read with its own stored norm; a cache of n such
 *     rows is tq_cache_bytes(TQ_FMT_TURBO4, 2n) bytes.  At d = 256 the write,
 *     dequantize and decode calls (one-call, staged and step) are available, for
 *     TURBO4 keys and values; prefill, the store, score output (scores_dbg) and the
 *     other formats return TQ_ERR_UNSUPPORTED.  Any other d returns
 *     TQ_ERR_UNSUPPORTED.
 *   - All functions return a tq_status; no exception crosses the ABI.
 *     tq_last_error() gives a one-line description of the last failure on the
 *     calling thread.
 *   - Device calls are asynchronous on the given stream (a cudaStream_t; NULL
 *     is the legacy default stream).  Arguments are validated on the host
 *     before any launch.  Launch failures map to TQ_ERR_CUDA.  Conditions only
 *     the device can see (a row id out of range, a sequence length outside
 *     [1, L], a bounded wait that ran out) are recorded in the context's
 *     device status word, read with tq_ctx_device_status().
 *   - A context belongs to the device that was current when it was created
 *     (its tables and status word live in that device's memory).  Every call
 *     that launches work, and every size query of the decode and prefill,
 *     checks that this device is the calling thread's current device and that
 *     the key and value contexts of the call belong to the same device;
 *     otherwise it returns TQ_ERR_INVALID_ARG and launches nothing.
 *   - The caller owns every device buffer (sources, caches, q, outputs,
 *     workspace).  The library owns only tq_ctx, which is immutable after
 *     creation and may be shared across streams.
 *   - Cache layout: rows of one packed record each, row r at byte r * row_bytes.
 *     For decode the cache is [B][Hkv][L] rows.  Cache base pointers must be
 *     16-byte aligned and the cache must be readable up to the next 16-byte
 *     boundary past its last row (tq_cache_bytes() returns that size).
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_HEAD_DIM 128

typedef struct CUstream_st *tq_stream_t; /* identical to cudaStream_t */
typedef struct tq_ctx tq_ctx;

typedef enum tq_status {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad enum, L == 0, ... */
  TQ_ERR_UNSUPPORTED = 2,  /* d not 128 / 256, format pair without a decode kernel, ... */
  TQ_ERR_ALIGNMENT = 3,    /* a pointer or stride breaks the stated alignment */
  TQ_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  TQ_ERR_ALLOC = 5,        /* device or host allocation failed */
  TQ_ERR_WORKSPACE = 6     /* workspace smaller than tq_decode_workspace_size() */
} tq_status;

/* Packed formats ([turbo4 post-mortem] sections 1, 4, 5, 7; [Triton deep dive] tricks 2-3).
 *   TURBO4  68 B/row: fp32 norm, qs[64]; 4-bit index j in bits 4*(j%2) of qs[j/2].
 *   TURBO3  56 B/row: four 14-B blocks {fp16 norm, qs[8], signs[4]}; index j of a
 *           block: low 2 bits at bits 2*(j%4) of qs[j/4], high bit at bit j%8 of
 *           signs[j/8]; each block carries the fp16 norm of the whole row.
 *   PROD3   56 B/row (keys): fp32 norm, fp32 residual norm, qs[32] 2-bit MSE
 *           indices (bits 2*(j%4) of byte j/4), signs[16] QJL bits (bit i%8 of
 *           byte i/8, 1 = +1).
 *   VGROUP2 48 B/row (values): q[32] 2-bit codes (bits 2*(j%4) of byte j/4),
 *           then 4 x {fp16 scale, fp16 zero} for groups of 32; value = code*scale+zero.
 * Every header is little-endian and comes first. */
typedef enum tq_format {
  TQ_FMT_TURBO4 = 0,
  TQ_FMT_TURBO3 = 1,
  TQ_FMT_PROD3 = 2,
  TQ_FMT_VGROUP2 = 3
} tq_format;

/* Codebook construction for the rotated-coordinate law N(0, 1/d).
 *   QUANTILE: conditional means of 2^bits equal-probability cells (reproduces the
 *             printed 16-entry d=128 table, [turbo4 post-mortem] section 5).
 *   LLOYD:    converged Lloyd-Max from the QUANTILE start ([turbo4 post-mortem]
 *             sections 5, 9; [Triton deep dive] "write path and codebook").
 *   DEFAULT:  QUANTILE for TURBO4, LLOYD for TURBO3 and PROD3. */
typedef enum tq_codebook_kind {
  TQ_CB_DEFAULT = 0,
  TQ_CB_QUANTILE = 1,
  TQ_CB_LLOYD = 2,
  TQ_CB_SPHERE = 3    /* Lloyd-Max under the exact law of a rotated unit-vector coordinate:
                         (1 + x)/2 ~ Beta((d-1)/2, (d-1)/2) ([Triton deep dive] "write path
                         and codebook": Lloyd-Max centroids for the rotated Beta law) */
} tq_codebook_kind;

/* Rotation y = R u applied before quantization.
 *   WHT:   R = (1/sqrt(d)) H D, D a seeded +-1 diagonal, H Sylvester Hadamard
 *          ([turbo4 post-mortem] sections 1, 10).
 *   DENSE: R = Pi, the Q factor (diag(R) > 0) of a seeded Gaussian d x d matrix
 *          ([Triton deep dive] trick 1), stored in fp32.
 * Randomness: splitmix64 outputs of the seed; WHT sign j = -1 when the top bit of
 * output j is set; Gaussians by Box-Muller on output pairs (row-major). */
typedef enum tq_rotation_kind {
  TQ_ROT_WHT = 0,
  TQ_ROT_DENSE = 1
} tq_rotation_kind;

typedef enum tq_dtype {
  TQ_DTYPE_F32 = 0,
  TQ_DTYPE_BF16 = 1,
  TQ_DTYPE_F16 = 2
} tq_dtype;

typedef struct tq_params {
  int32_t d;          /* must be 128 */
  int32_t format;     /* tq_format */
  int32_t codebook;   /* tq_codebook_kind (ignored for VGROUP2) */
  int32_t rotation;   /* tq_rotation_kind (ignored for VGROUP2, which is not rotated) */
  uint64_t rot_seed;  /* seed of the rotation */
  uint64_t qjl_seed;  /* seed of the QJL matrix S (PROD3 only; must differ from rot_seed,
                         [turbo4 post-mortem] section 10) */
  int32_t qjl_shrink; /* PROD3 reads: 0 = the unbiased estimator (sqrt(pi/2)/d) gamma S^T sigma,
                         1 = that term times 2/pi ([turbo4 post-mortem] section 3's shrinkage).
                         The stored bytes do not depend on it. */
  int32_t reserved;   /* must be 0 */
} tq_params;

/* ---------------------------------------------------------------- host only */

/* Codebook of 2^bits centroids and 2^bits - 1 decision boundaries for N(0, 1/d),
 * built in fp64 and rounded to fp32; boundaries are the fp32 rounding of the
 * midpoints of adjacent stored centroids.  bits in 1..4, d == 128, kind QUANTILE
 * or LLOYD.  centroids: host array of 2^bits floats; boundaries: host array of
 * 2^bits - 1 floats (may be NULL).  Caller-owned.  No device work. */
tq_status tq_make_codebook(int bits, int d, int kind, float *centroids, float *boundaries);

/* The seeded rotation as host data.  DENSE: out is d*d floats, row-major Pi
 * (y = Pi u).  WHT: out is d floats, the diagonal D (+1/-1).  No device work. */
tq_status tq_make_rotation(int kind, int d, uint64_t seed, float *out);

/* The QJL matrix S (d*d floats, row-major, i.i.d. N(0,1) from `seed`).  No device work. */
tq_status tq_make_qjl_matrix(int d, uint64_t seed, float *out);

/* Bytes of one packed row of `format` (68, 56, 56, 48); -1 for a bad format. */
int64_t tq_row_bytes(int format);

/* Bytes a cache of n_rows rows must provide: n_rows * row_bytes rounded up to 16. */
size_t tq_cache_bytes(int format, int64_t n_rows);

const char *tq_status_string(tq_status s);
const char *tq_last_error(void);

/* ------------------------------------------------------------- context / device */

/* Builds codebook, rotation and (PROD3) QJL matrix on the current CUDA device.
 * *out receives a context owned by the library; free it with tq_ctx_destroy(). */
tq_status tq_ctx_create(const tq_params *params, tq_ctx **out);
tq_status tq_ctx_destroy(tq_ctx *ctx);

/* Reads (synchronising the device) and optionally clears the context's device
 * status word: 0 = no device-side error; 1 = row id out of range (write skipped);
 * 2 = sequence length outside [1, L] (clamped); 3 = a bounded wait ran out;
 * 4 = the decode kernel found shared memory laid out unlike the device reported
 * (no output was computed). */
tq_status tq_ctx_device_status(const tq_ctx *ctx, int32_t *status, int clear);

/* Write path / SET_ROWS ([turbo4 post-mortem] sections 1, 2): quantize n_rows
 * source rows of 128 elements and store packed row i at cache slot row_ids[i].
 *   src            device, n_rows rows of src_dtype (F32 or BF16), row i at
 *                  src + i * src_row_stride elements.  BF16 rows must be 8-byte
 *                  aligned, F32 rows 16-byte aligned.
 *   row_ids        device int64[n_rows] cache slots, or NULL for slot i.
 *   dst_cache      device, dst_rows packed rows of ctx's format (16-byte aligned).
 * Rows whose slot is outside [0, dst_rows) are skipped and flagged (status 1).
 * n_rows == 0 is a no-op.  Rows of the same slot written twice race. */
tq_status tq_quantize_set_rows(const tq_ctx *ctx, const void *src, int src_dtype,
                               int64_t n_rows, int64_t src_row_stride,
                               const int64_t *row_ids, void *dst_cache, int64_t dst_rows,
                               tq_stream_t stream);

/* Dequantize ([turbo4 post-mortem] section 4; [Triton deep dive] "hybrid" path):
 * dst[i] = reconstruction of packed row i, fp32 [n_rows][128] (device).  With
 * unrotate != 0 the rotated formats are mapped back by R^T; with 0 they return
 * the rotated-basis values norm * c[idx] (PROD3 and VGROUP2 always reconstruct
 * the original space). */
tq_status tq_dequantize(const tq_ctx *ctx, const void *cache, int64_t n_rows, int unrotate,
                        float *dst, tq_stream_t stream);

/* Decode attention ([Triton deep dive] tricks 1-3): for batch b and q-head h,
 * with KV head kv = floor(h * Hkv / Hq),
 *   out[b,h] = sum_t softmax_t(scale * <q[b,h], K_hat[b,kv,t]>) V_hat[b,kv,t],
 * t < seq_lens[b], computed from the packed caches without materialising K/V:
 * q is rotated (and, for PROD3 keys, sketched with S) once, every key is scored
 * from its indices, online softmax runs split-K across SMs, values are
 * dequantized in registers, and the output is un-rotated once per head.
 *   k_ctx / v_ctx  contexts of the key and value caches.  Supported pairs:
 *                  (TURBO4, TURBO4); (TURBO3, TURBO4) -- the asymmetric 3-bit-key /
 *                  4-bit-value cache of [turbo4 post-mortem] section 9; (TURBO3,
 *                  TURBO3) -- the 3.5-bit cache of its section 1; (TURBO4, TURBO3);
 *                  (PROD3, VGROUP2).  Every 32-element TURBO3 block, key or value, is
 *                  scaled by its own stored norm.
 *   q              device [B][Hq][128] of q_dtype (F32, BF16 or F16), 16-byte aligned.
 *   k_cache/v_cache device [B][Hkv][L] packed rows.
 *   seq_lens       device int32[B] lengths in [1, L], or NULL for all L.
 *   scale          softmax scale; 0 selects 1/sqrt(128).
 *   out            device fp32 [B][Hq][128].
 *   scores_dbg     NULL, or device fp32 [B][Hq][L]: the scaled scores (tests).
 *   workspace      device scratch of at least tq_decode_workspace_size() bytes,
 *                  256-byte aligned; its contents need no initialisation.
 * Hq must be a multiple of Hkv.  L >= 1, B >= 1.
 * Launches: the q preparation, the split-K kernel and, unless the split-K kernel
 * merges the splits itself (the CTA that completes a (batch, KV head, head group)
 * unit merges its partials, un-rotates and writes the unit's outputs; TURBO4 /
 * TURBO3 keys and values when each CTA completes few units), the combine kernel;
 * tq_decode_num_launches tells which for a shape. */
tq_status tq_decode_workspace_size(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int Hq,
                                   int Hkv, int L, size_t *bytes);
/* One decode step ([turbo4 post-mortem] §1-§2 for the row writes, [Triton deep dive]
 * tricks 1-3 for the decode): append the step's new K and V rows (SET_ROWS of new_k
 * into k_cache and new_v into v_cache, n_rows rows each at slots row_ids of the
 * [B][Hkv][L] caches, as tq_quantize_set_rows), then tq_decode_attention over the
 * updated caches.  The same results as those three calls; for TURBO4 / TURBO3 caches
 * (both under the dense or both under the WHT rotation), or PROD3 keys with VGROUP2
 * values, and at most 256 rows, the two writes and the q preparation share one launch
 * (they are independent), so the step has one wait on the previous kernel where the
 * three calls have three.  Arguments as in tq_quantize_set_rows (dst_rows =
 * B * Hkv * L; new_k and new_v share src_dtype and src_row_stride) and
 * tq_decode_attention (no scores); every buffer is the caller's device memory, used in
 * stream order.  Errors: all the checks of the three calls are made before anything is
 * launched (TQ_ERR_INVALID_ARG, TQ_ERR_ALIGNMENT, TQ_ERR_UNSUPPORTED, TQ_ERR_WORKSPACE);
 * a slot outside the caches is skipped and flagged in the context's device status, as
 * in tq_quantize_set_rows. */
tq_status tq_decode_step(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *new_k,
                         const void *new_v, int src_dtype, int64_t n_rows, int64_t src_row_stride,
                         const int64_t *row_ids, const void *q, int q_dtype, void *k_cache,
                         void *v_cache, const int32_t *seq_lens, int B, int Hq, int Hkv, int L,
                         float scale, float *out, void *workspace, size_t workspace_bytes,
                         tq_stream_t stream);
/* tq_decode_step with host buffers: the step's new K / V rows and q are copied in one
 * piece from host memory into the caller's device staging area, tq_decode_step runs on
 * them, and the output is copied back to host memory -- all enqueued on `stream`; the call
 * returns without waiting (synchronize the stream before reading out_host).  Host buffers
 * should be pinned (page-locked) for the copies to be asynchronous.
 *   inputs_host    one host buffer: the n_rows new K rows [n_rows][d] of src_dtype (F32 or
 *                  BF16), then the n_rows new V rows, then q [B][Hq][d] of q_dtype, back to
 *                  back; d = k_ctx's head dimension.
 *   out_host       host fp32 [B][Hq][d].
 *   staging        device scratch of at least tq_decode_step_host_staging_size() bytes,
 *                  256-byte aligned: the inputs and the output on the device.
 *   the rest       as tq_decode_step (row_ids, caches, seq_lens, workspace: device).
 * In place: when inputs_host and out_host are each one page-locked allocation
 * (cudaHostAlloc / cudaMallocHost) mapped for the current device, inputs_host 16-byte
 * and out_host 4-byte aligned, the head dimension 128 and n_rows <= 256, no copy is
 * issued: the step's kernels read the inputs from and write the output to host memory
 * directly (coherent over the chip-to-chip link on GB300), and the staging area is not
 * used.  The host checks both ends of each range before taking this path.
 * Errors: the checks of the staging, the shape and the workspace come before the copy;
 * the remaining checks are tq_decode_step's (made before it launches anything; the input
 * copy has then already been enqueued, into the staging area only). */
tq_status tq_decode_step_host(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *inputs_host, int src_dtype,
                              int64_t n_rows, const int64_t *row_ids, int q_dtype, void *k_cache, void *v_cache,
                              const int32_t *seq_lens, int B, int Hq, int Hkv, int L, float scale,
                              float *out_host, void *staging, size_t staging_bytes, void *workspace,
                              size_t workspace_bytes, tq_stream_t stream);
/* Bytes of device staging tq_decode_step_host needs for these inputs. */
tq_status tq_decode_step_host_staging_size(const tq_ctx *k_ctx, int src_dtype, int64_t n_rows, int q_dtype,
                                           int B, int Hq, size_t *bytes);
/* Number of kernels tq_decode_step launches for these arguments: 2 or 3 on the one-launch
 * front (see above), else 2 more for the two writes (none when n_rows == 0). */
tq_status tq_decode_step_num_launches(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int src_dtype,
                                      int64_t n_rows, int B, int Hq, int Hkv, int L, int *n);
/* Number of kernels tq_decode_attention launches for this shape (2 or 3). */
tq_status tq_decode_num_launches(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int Hq,
                                 int Hkv, int L, int *n);
tq_status tq_decode_attention(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *q,
                              int q_dtype, const void *k_cache, const void *v_cache,
                              const int32_t *seq_lens, int B, int Hq, int Hkv, int L,
                              float scale, float *out, float *scores_dbg, void *workspace,
                              size_t workspace_bytes, tq_stream_t stream);

/* The three stages of tq_decode_attention, for callers that time or overlap them;
 * same arguments and workspace, run in this order on one stream:
 *   prepare_q: q_rot = R q (and S q), pre-scaled and split for the tensor cores;
 *   partial:   split-K scan of the packed caches -> per-split (max, sum, acc);
 *   combine:   log-sum-exp merge of the splits, 1/sum, un-rotation, write out. */
tq_status tq_decode_prepare_q(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *q,
                              int q_dtype, int B, int Hq, int Hkv, int L, float scale,
                              void *workspace, size_t workspace_bytes, tq_stream_t stream);
tq_status tq_decode_partial(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *k_cache,
                            const void *v_cache, const int32_t *seq_lens, int B, int Hq,
                            int Hkv, int L, float *scores_dbg, void *workspace,
                            size_t workspace_bytes, tq_stream_t stream);
tq_status tq_decode_combine(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int Hq, int Hkv,
                            int L, float *out, void *workspace, size_t workspace_bytes,
                            tq_stream_t stream);

/* Stages two and three of tq_decode_attention in one call, as tq_decode_attention
 * runs them: the split-K decode with the merge and the un-rotation done inside the
 * split-K kernel where the shape allows it (one launch), else the split-K kernel and
 * the combine kernel (tq_decode_num_launches() - 1 launches either way).  The
 * workspace must hold tq_decode_prepare_q's output for the same shape; the per-unit
 * counters of the fused merge are zeroed there and every completed call leaves them
 * zero again, so the call may be repeated over the same prepared q.  Arguments and
 * errors as tq_decode_attention (no q, scale or scores). */
tq_status tq_decode_partial_merge(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *k_cache,
                                  const void *v_cache, const int32_t *seq_lens, int B, int Hq, int Hkv,
                                  int L, float *out, void *workspace, size_t workspace_bytes,
                                  tq_stream_t stream);

/* Chunked prefill attention over the compressed cache ([turbo4 post-mortem] §9,
 * the prefill table: a prompt is processed in chunks that attend to the turbo4
 * cache, which already holds the chunk's own rows -- write them with
 * tq_quantize_set_rows first).  For batch b, chunk query i (0 <= i < T) and q-head
 * h, with KV head kv = floor(h * Hkv / Hq) and position p = q_start[b] + i,
 *   out[b,i,h] = sum_{t <= p} softmax_t(scale * <q[b,i,h], K_hat[b,kv,t]>) V_hat[b,kv,t]
 * (causal: keys after the query's own position are not attended).  q is rotated
 * once, scores and the PV product run as tensor-core products over fp16 operands
 * decoded from the packed tiles, online softmax per row, split over the SMs, and
 * the output is un-rotated once per row.
 *   k_ctx / v_ctx  TURBO4 contexts (others: TQ_ERR_UNSUPPORTED).
 *   q              device [B][T][Hq][128] of q_dtype (F32, BF16 or F16), 16-byte aligned.
 *   k_cache/v_cache device [B][Hkv][L] packed rows, 16-byte aligned.
 *   q_start        device int32[B]: position of query 0 of each sequence; must lie
 *                  in [0, L - T] (outside: clamped and flagged, device status 2).
 *   scale          softmax scale; 0 selects 1/sqrt(128).
 *   out            device fp32 [B][T][Hq][128].
 *   workspace      device scratch of tq_prefill_workspace_size() bytes, 256-byte
 *                  aligned, no initialisation needed.
 * Hq / Hkv must divide 128 (the rows of a tile are 128 / (Hq/Hkv) queries of all the
 * KV head's q-heads); 1 <= T <= L.  The work is split evenly over all of L's key
 * tiles, so pass the smallest L that covers the attended keys. */
tq_status tq_prefill_workspace_size(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int T, int Hq,
                                    int Hkv, int L, size_t *bytes);
tq_status tq_prefill_attention(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *q, int q_dtype,
                               const void *k_cache, const void *v_cache, const int32_t *q_start,
                               int B, int T, int Hq, int Hkv, int L, float scale, float *out,
                               void *workspace, size_t workspace_bytes, tq_stream_t stream);

/* The three stages of tq_prefill_attention (same arguments and workspace, in this
 * order on one stream): q rotation and split; the tensor-core scan of the packed
 * caches -> per-split (max, sum, O) per row; merge, 1/sum and un-rotation. */
tq_status tq_prefill_prepare_q(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *q, int q_dtype,
                               int B, int T, int Hq, int Hkv, int L, float scale, void *workspace,
                               size_t workspace_bytes, tq_stream_t stream);
tq_status tq_prefill_partial(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *k_cache,
                             const void *v_cache, const int32_t *q_start, int B, int T, int Hq,
                             int Hkv, int L, void *workspace, size_t workspace_bytes,
                             tq_stream_t stream);
tq_status tq_prefill_combine(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int T, int Hq, int Hkv,
                             int L, float *out, void *workspace, size_t workspace_bytes,
                             tq_stream_t stream);

/* ---------------------------------------------------------- capture + store */

/* Ring-buffer capture and block-append store ([Triton deep dive] "write path and
 * codebook": a ring buffer holds the most recent exact tokens; when it is full the
 * oldest batch is compressed into the cache, so the decode hot path quantizes
 * nothing per token; the store appends by blocks).  One store holds B sequences of
 * Hkv KV heads, all of the same length:
 *   tokens [0, flushed)   compressed rows in the store's caches [B][Hkv][L];
 *   tokens [flushed, len) exact bf16 rows in a ring of ring_tokens slots.
 * When an append finds the ring full, the oldest ring_tokens/2 tokens of every
 * (sequence, KV head) are quantized by one SET_ROWS launch per cache and flushed
 * advances by ring_tokens/2; tq_store_decode attends over both parts (split-K
 * decode over the compressed prefix, one exact partial over the ring, one merge).
 * All calls of one store must use one stream; the host-side counters advance with
 * each call, the device work runs in stream order.  The store owns its device
 * memory (caches, ring, flush indices), freed by tq_store_destroy. */
typedef struct tq_store tq_store;

/*   k_ctx / v_ctx  a supported decode pair (see tq_decode_attention), on the
 *                  current device; the store keeps the pointers (contexts outlive it).
 *   L              compressed capacity per sequence (tokens).
 *   ring_tokens    even, 2..4096: exact tokens kept; blocks of ring_tokens/2 are flushed. */
tq_status tq_store_create(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int Hkv, int L,
                          int ring_tokens, tq_store **out);
tq_status tq_store_destroy(tq_store *store);

/* Append n tokens to every sequence: k_new / v_new device bf16 [B][Hkv][n][128],
 * 16-byte aligned.  TQ_ERR_INVALID_ARG (and nothing appended) when the flushes the
 * append needs would pass L. */
tq_status tq_store_append(tq_store *store, const void *k_new, const void *v_new, int n,
                          tq_stream_t stream);

/* Host-side state: tokens per sequence, compressed tokens, and the device caches
 * (packed rows [B][Hkv][L]; rows at or past `flushed` are not yet meaningful).
 * Any output pointer may be NULL. */
tq_status tq_store_state(const tq_store *store, int64_t *len, int64_t *flushed,
                         const void **k_cache, const void **v_cache);

/* Decode over the whole store: q device [B][Hq][128] of q_dtype (F32, BF16, F16),
 * 16-byte aligned; out device fp32 [B][Hq][128]; scale 0 selects 1/sqrt(128);
 * workspace of tq_store_workspace_size() bytes, 256-byte aligned.  Hq must be a
 * multiple of Hkv.  The store must hold at least one token. */
tq_status tq_store_workspace_size(const tq_store *store, int Hq, size_t *bytes);
tq_status tq_store_decode(const tq_store *store, const void *q, int q_dtype, int Hq, float scale,
                          float *out, void *workspace, size_t workspace_bytes, tq_stream_t stream);

/* Number of key splits the decode uses for this shape on the current device. */
tq_status tq_decode_num_splits(const tq_ctx *k_ctx, const tq_ctx *v_ctx, int B, int Hq,
                               int Hkv, int L, int *n_split);

/* tq_decode_attention without a workspace argument and without any allocation.
 * The method's pages have no counterpart: this is a deployment variant of the
 * same fused decode, with identical arithmetic and outputs.
 *
 * For callers that can neither allocate device memory nor hand over a
 * workspace: plugin code inside a host framework that owns and accounts for
 * all device memory, and step loops where cudaMalloc / cudaFree could wait for
 * the whole device.  The scratch (rotated queries, split-K partials) lives in
 * a static device array of TQ_STATIC_WORKSPACE_BYTES that the library's module
 * carries on each device; the call performs no allocation of any kind.
 *
 * Arguments: as tq_decode_attention (no scores_dbg, workspace or size).
 * Errors: TQ_ERR_WORKSPACE when the shape needs more scratch than
 *   TQ_STATIC_WORKSPACE_BYTES (tq_decode_workspace_size() tells; such shapes
 *   use tq_decode_attention); the other errors of tq_decode_attention.
 * Set-up: the contexts' device must be current (as for every call).  The first
 *   call on each device looks up the static area's address there once, which
 *   may load the module on that device; make that first call before any other
 *   work that must not be interrupted by module loading.
 * Nothing in the area needs to start at zero: every word the decode reads is
 *   written earlier in the same call.
 * Concurrency: all calls on one device share the single area.  Two calls whose
 *   executions overlap on the device (different streams, or otherwise not
 *   ordered) race on it and give wrong results; order them on one stream. */
#define TQ_STATIC_WORKSPACE_BYTES (4u << 20)
tq_status tq_decode_attention_static(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *q,
                                     int q_dtype, const void *k_cache, const void *v_cache,
                                     const int32_t *seq_lens, int B, int Hq, int Hkv, int L,
                                     float scale, float *out, tq_stream_t stream);
/* TQ_STATIC_WORKSPACE_BYTES as compiled into the library (bindings read it here). */
size_t tq_static_workspace_bytes(void);

/* ------------------------------------------------------------- testing hook */

/* Failure detection test (no counterpart on the pages): runs the split-K decode
 * kernel of tq_decode_partial (TURBO4 pair) with its producer withholding the first
 * tile, so every consumer's bounded wait runs out (about 2 s).  The kernel then
 * records status 3 in k_ctx's status word and returns without output; the context
 * and the device stay usable.  Arguments as tq_decode_partial (no seq_lens, no
 * scores); nothing is written to the caches. */
tq_status tq_test_decode_wait_timeout(const tq_ctx *k_ctx, const tq_ctx *v_ctx, const void *k_cache,
                                      const void *v_cache, int B, int Hq, int Hkv, int L, void *workspace,
                                      size_t workspace_bytes, tq_stream_t stream);

/* Device-check test (no counterpart on the pages): overwrites the device a context
 * is recorded to belong to, so a test on a one-GPU machine can make the
 * current-device check of every launching call fail (TQ_ERR_INVALID_ARG, nothing
 * launched) and then restore the true device.  Not for use outside tests. */
tq_status tq_test_ctx_set_device(tq_ctx *ctx, int device);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
