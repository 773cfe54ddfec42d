// Device helpers: inline PTX wrappers (byte permute, legacy-register tensor-core
// MMA, mbarrier, bulk async copy) and small numeric utilities.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace tq {

constexpr unsigned FULL_MASK = 0xffffffffu;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 8 packed 4-bit indices of a symmetric 16-entry codebook -> 8 fp16 centroid values as
// four fp16x2 words; lo / hi are the byte planes of the eight magnitudes (F16Table).
// Magnitude index m = idx for idx < 8 (negative centroids), 15 - idx otherwise;
// sign is negative when bit 3 of the index is clear.  SEL0 / SEL1 choose how the
// looked-up bytes pair up: (0,1),(2,3) for dims of one key, (0,2),(1,3) for the
// same dim of two keys after a byte interleave.
template <uint32_t SEL0, uint32_t SEL1>
__device__ __forceinline__ void decode8(uint32_t x, const uint32_t (&lo)[2],
                                        const uint32_t (&hi)[2], uint32_t (&r)[4]) {
  const uint32_t t = x & 0x88888888u;
  const uint32_t m = (x ^ (t - (t >> 3))) & 0x77777777u;
  const uint32_t x4 = x << 4;
  const uint32_t pos_a = prmt(x, x4, 0x9D8Cu);  // 0xFF per byte where nibble 0..3 >= 8
  const uint32_t pos_b = prmt(x, x4, 0xBFAEu);  // nibbles 4..7
  const uint32_t mh = m >> 16;
  const uint32_t lo_a = prmt(lo[0], lo[1], m);
  const uint32_t lo_b = prmt(lo[0], lo[1], mh);
  const uint32_t hi_a = prmt(hi[0], hi[1], m) | (~pos_a & 0x80808080u);
  const uint32_t hi_b = prmt(hi[0], hi[1], mh) | (~pos_b & 0x80808080u);
  r[0] = prmt(lo_a, hi_a, SEL0);
  r[1] = prmt(lo_a, hi_a, SEL1);
  r[2] = prmt(lo_b, hi_b, SEL0);
  r[3] = prmt(lo_b, hi_b, SEL1);
}

// D += A * B for one m16n8k16 tile, fp16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);  // .x (low 16 bits) = lo
  return *reinterpret_cast<uint32_t *>(&h);
}

// Split two fp32 values into fp16 hi + lo pairs (hi = RN(x), lo = RN(x - hi)).
__device__ __forceinline__ void split_half2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  __half2 h = __floats2half2_rn(x0, x1);
  float2 hf = __half22float2(h);
  __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<uint32_t *>(&h);
  lo = *reinterpret_cast<uint32_t *>(&l);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float log2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Index of the nearest centroid, #{k : y > b_k}, from the grid table (see BucketTable);
// cnt, e: the table's arrays staged in shared memory.
__device__ __forceinline__ uint32_t bucket_grid(float y, float scale, float offset, int n,
                                                const uint8_t *cnt, const float *e) {
  int t = __float2int_rd(fmaf(y, scale, offset));  // NaN -> 0, +-inf -> saturated
  t = min(max(t, 0), n - 1);
  return (uint32_t)cnt[t] + (y > e[t] ? 1u : 0u);
}

// ---- programmatic dependent launch ----
// Every kernel of the library is launched so that it may start while the previous
// kernel on the stream is still finishing: it runs its prologue (work that reads only
// the immutable context), then waits here until the previous grid has completed and its
// memory is visible.  Without such a launch the wait returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allows the next kernel on the stream to be scheduled (it still waits in pdl_wait for
// this grid to complete before touching its results).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- mbarrier + bulk async copy (shared::cta barriers, CTA-local copies) ----

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One attempt; the thread may sleep up to about 20 us inside it (suspend-time hint)
// and wakes as soon as the phase completes, so a waiting warp issues few instructions.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 20000;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after `limit_ns` of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 4; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
// Prefetch `bytes` (a multiple of 16, 16-byte aligned source) into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

}  // namespace tq
