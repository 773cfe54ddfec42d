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
// the next unit's q), and the sched_v virtual tiles are split over the sched_g CTAs in
// proportion: CTA c takes [c * sched_v / sched_g, (c + 1) * sched_v / sched_g), rounded
// down, so the ranges differ by at most one tile and a CTA whose range crosses into
// another unit gets fewer real tiles.  vx = 0 is an equal split of the real tiles.
struct Item {
  int unit, t0, t1, slot;  // tiles [t0, t1) of the unit; partial slot of this CTA
};

// The schedule arithmetic runs in 32 bits: the host checks vtotal < 2^31 and
// grid^2 < 2^31 and stores V / G, V % G and two float reciprocals (set_schedule), so no
// 64-bit division sits on a CTA's path (each took several hundred cycles at the start of
// an item and in the fused merge).

// Start of CTA c's virtual range, floor(c * V / G) for 0 <= c <= G: c * (V / G) plus
// floor(c * (V % G) / G), the second from a float estimate that is within one of it.
template <typename P>
__device__ __forceinline__ int sched_start(const P &p, int c) {
  const uint32_t G = (uint32_t)p.sched_g;
  const uint32_t x = (uint32_t)c * p.sched_r;  // < G^2 < 2^31
  uint32_t t = __float2uint_rz((float)x * p.sched_ginv);
  if (t * G > x)
    --t;
  else if ((t + 1) * G <= x)
    ++t;
  return (int)((uint32_t)c * p.sched_q + t);
}

// First real tile at or after virtual position v (0 <= v <= V).
template <typename P>
__device__ __forceinline__ int real_tile(const P &p, int v) {
  const uint32_t vu = (uint32_t)(p.vx + p.tiles_per_unit);
  const uint32_t u = (uint32_t)v / vu;
  const int o = v - (int)(u * vu) - p.vx;
  return (int)u * p.tiles_per_unit + (o > 0 ? o : 0);
}
template <typename P>
__device__ __forceinline__ int cta_first_tile(const P &p, int cta) {
  return min(real_tile(p, sched_start(p, cta)), p.total_tiles);
}
// The CTA whose range holds virtual tile v (0 <= v < V): the largest c < G with
// sched_start(c) <= v.  A float estimate of v * G / V lies within two of it; the
// monotone steps below end on the exact value.
template <typename P>
__device__ __forceinline__ int cta_of_vtile(const P &p, int v) {
  int c = min(max(__float2int_rz((float)v * p.sched_inv), 0), p.sched_g - 1);
  while (c > 0 && sched_start(p, c) > v) --c;
  while (c + 1 < p.sched_g && sched_start(p, c + 1) <= v) ++c;
  return c;
}
// CTAs whose range meets unit u: unit_first_cta(u) .. + unit_n_split(u) - 1.
template <typename P>
__device__ __forceinline__ int unit_first_cta(const P &p, int u) {
  return cta_of_vtile(p, u * (p.vx + p.tiles_per_unit) + p.vx);
}
template <typename P>
__device__ __forceinline__ int unit_n_split(const P &p, int u) {
  const int v0 = u * (p.vx + p.tiles_per_unit) + p.vx;
  return cta_of_vtile(p, v0 + p.tiles_per_unit - 1) - cta_of_vtile(p, v0) + 1;
}

// Host: the schedule's fields of a kernel's parameters (grid G CTAs over V virtual
// tiles).  False when the 32-bit arithmetic above does not hold for these sizes.
template <typename P>
inline bool set_schedule(P &p, int grid, int64_t vtotal) {
  if (grid < 1 || vtotal < grid || vtotal > INT32_MAX || (int64_t)grid * grid > INT32_MAX) return false;
  p.sched_g = grid;
  p.sched_v = (int)vtotal;
  p.sched_q = (uint32_t)(vtotal / grid);
  p.sched_r = (uint32_t)(vtotal % grid);
  p.sched_ginv = 1.0f / (float)grid;
  p.sched_inv = (float)grid / (float)vtotal;
  return true;
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

// CTA-wide barrier 0 of N threads, split: the producer warp arrives without waiting, the
// consumer warps wait for every thread (the producer's shared-memory writes before its
// arrive are visible to them afterwards).
template <int N>
__device__ __forceinline__ void named_arrive0() {
  asm volatile("bar.arrive 0, %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void named_sync0() {
  asm volatile("bar.sync 0, %0;" ::"n"(N) : "memory");
}

}  // namespace tq
