// Pieces shared by the split-K decode kernels: numeric constants of the online
// softmax, the persistent tile schedule (units laid end to end, one contiguous tile
// range per CTA) and the shared-window placement of the decode tables.
#pragma once

#include <stdint.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

constexpr float P_SHIFT = 7.0f;        // p' = 2^7 * exp2(.) keeps the fp16 operand normal
constexpr float RESCALE_SLACK = 8.0f;  // rescale only when the max grows by more than 2^8,
                                       // so p' <= 2^(7+8) stays inside fp16
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr uint32_t LUT_WINDOW = 0x10000;  // shared-window address of a 64 KB decode table
constexpr uint32_t RESERVED_SMEM = 1024;  // window bytes before dynamic smem (usual value)

// Work item = the tiles of one unit (batch, KV head, head group) inside this CTA's
// contiguous range of the global tile sequence; units are laid end to end, so a CTA
// touches at most a few units and each (unit, CTA) pair gives one partial.
//
// Cost-balanced ranges: each unit counts vx virtual tiles ahead of its tiles_per_unit
// real ones (the fixed cost of one more item: the warps' merge, the partial's write,
// the next unit's q), and every CTA takes tiles_per_cta tiles of that virtual sequence,
// so a CTA whose range crosses into another unit gets fewer real tiles.  vx = 0 is an
// equal split of the real tiles.
struct Item {
  int unit, t0, t1, slot;  // tiles [t0, t1) of the unit; partial slot of this CTA
};

// First real tile at or after virtual position v.
template <typename P>
__device__ __forceinline__ int real_tile(const P &p, int64_t v) {
  const int64_t vu = (int64_t)p.vx + p.tiles_per_unit;
  const int64_t u = v / vu;
  const int64_t o = v - u * vu - p.vx;
  return (int)(u * p.tiles_per_unit + (o > 0 ? o : 0));
}
template <typename P>
__device__ __forceinline__ int cta_first_tile(const P &p, int cta) {
  return min(real_tile(p, (int64_t)cta * p.tiles_per_cta), p.total_tiles);
}
// CTAs whose range meets unit u: unit_first_cta(u) .. + unit_n_split(u) - 1.
template <typename P>
__device__ __forceinline__ int unit_first_cta(const P &p, int u) {
  return (int)(((int64_t)u * (p.vx + p.tiles_per_unit) + p.vx) / p.tiles_per_cta);
}
template <typename P>
__device__ __forceinline__ int unit_n_split(const P &p, int u) {
  const int64_t v0 = (int64_t)u * (p.vx + p.tiles_per_unit) + p.vx;
  return (int)((v0 + p.tiles_per_unit - 1) / p.tiles_per_cta - v0 / p.tiles_per_cta + 1);
}

template <typename P>
__device__ __forceinline__ bool next_item(const P &p, int cta, int &t, Item &it) {
  const int end = cta_first_tile(p, cta + 1);
  if (t >= end) return false;
  it.unit = t / p.tiles_per_unit;
  it.t0 = t - it.unit * p.tiles_per_unit;
  it.t1 = min(end - it.unit * p.tiles_per_unit, p.tiles_per_unit);
  it.slot = cta - unit_first_cta(p, it.unit);
  t += it.t1 - it.t0;
  return true;
}

// Keys of the unit's sequence: seq_lens[b] clamped to [1, L] (L without seq_lens).
template <typename P>
__device__ __forceinline__ int unit_len(const P &p, int unit) {
  const int b = unit / (p.Hkv * p.n_hg);
  if (!p.seq_lens) return p.L;
  const int v = p.seq_lens[b];
  return v < 1 ? 1 : (v > p.L ? p.L : v);
}

// Barrier over the first N threads (the consumer warps; the producer never joins).
template <int N>
__device__ __forceinline__ void named_sync1() {
  asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

}  // namespace tq
