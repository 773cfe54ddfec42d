// 5th-generation tensor-core helpers (tcgen05 with tensor-memory accumulators) shared by
// the tensor-core write and the prefill attention: the 128-byte swizzled K-major
// shared-memory operand layout and its matrix descriptor, instruction descriptors,
// tensor-memory allocation, the MMA issue / commit, and 32-column loads and stores of
// one accumulator lane.
#pragma once

#include <stdint.h>

#include "tq_device.cuh"

namespace tq {

constexpr uint32_t SW_ROWS = 128;                     // rows of an operand tile (M or N)
constexpr uint32_t SW_HALF_BYTES = SW_ROWS * 128;     // one 64-column half of a 16-bit tile
constexpr uint32_t SW_TILE_BYTES = 2 * SW_HALF_BYTES; // 128 x 128 16-bit elements, 32 KB

// Offset of element (row, k) of a 128 x 128 16-bit tile in the 128-byte swizzled
// K-major layout: two halves of 64 columns, rows of 128 bytes, 16-byte chunk c of row r
// stored at chunk position c ^ (r % 8).  The tile base must be 1024-byte aligned.
__host__ __device__ constexpr uint32_t sw128_offset(uint32_t row, uint32_t k) {
  return (k >> 6) * SW_HALF_BYTES + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + (k & 7) * 2;
}

// Shared-memory matrix descriptor of that layout: 128-byte swizzle, 8-row groups 1024
// bytes apart (the leading offset is unused for this layout).  K-step s of 16 elements
// starts at sw128_offset(0, 16 s): + 32 s bytes inside a half, + SW_HALF_BYTES per half.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;                         // leading byte offset (unused), 16 B
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // stride byte offset: 1024 B
  d |= (uint64_t)1 << 46;                         // descriptor version
  d |= (uint64_t)2 << 61;                         // 128-byte swizzle
  return d;
}
__device__ __forceinline__ uint32_t sw128_kstep(int s) {
  return (uint32_t)(s >> 2) * SW_HALF_BYTES + (uint32_t)(s & 3) * 32;
}

// Instruction descriptors of kind::f16, fp32 accumulator, both operands K-major,
// M = N = 128: bf16 A and B, or fp16 A and B (one MMA never mixes the two).
constexpr uint32_t IDESC_M128_N128 = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t IDESC_BF16 = IDESC_M128_N128 | (1u << 7) | (1u << 10);
constexpr uint32_t IDESC_F16 = IDESC_M128_N128;

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes made visible to the tensor core's operand reads.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D (tensor memory) = A B^T (+ D when accumulate != 0), A and B from shared memory.
template <uint32_t IDESC>
__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate));
}
// D (tensor memory) = A B^T (+ D when accumulate != 0), A from tensor memory (row m of A
// in lane m, two 16-bit K elements per 32-bit column, the lower K index in the low half;
// an MMA of K = 16 reads 8 columns from tmem_a), B from shared memory.
template <uint32_t IDESC>
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(IDESC), "r"(accumulate));
}
// The mbarrier completes when every MMA this thread issued so far has finished.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane (a warp reads the 32
// lanes of its quarter).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 32 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  tmem_st32(taddr, r);
}

}  // namespace tq
