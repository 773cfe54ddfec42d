/*
 * The CPU baseline of the decode benchmark: a plain fp32 compressed-domain decode loop
 * over turbo4 keys and values, parallel over (batch, KV head) units with OpenMP.
 *
 * Test and benchmark infrastructure only, like everything under oracle/: it is not the
 * oracle of any parity test (the oracle is the fp64 dequantize-then-softmax definition
 * in attention.py), it is what the benchmark times on the host cores beside the GPU.
 * It follows the algebra of "TurboQuant fused Triton kernels deep dive", tricks 1-3,
 * in plain scalar code:
 *   - rotate each query once, q_rot = R_K q (trick 1: <q, R^T y> = <R q, y>);
 *   - score every key from its indices: s = scale * n * sum_j q_rot[j] c[idx_j];
 *   - single-pass online softmax over the keys (running max m, sum l, accumulator);
 *   - accumulate values in their rotated basis, acc += p * n_v * c_V[idx_j] (trick 3);
 *   - one un-rotation of the output per head, o = R_V^T (acc / l).
 * The turbo4 record (post-mortem "how the turbo4 KV format came back", sections 5 and
 * 7): fp32 norm in bytes 0-3, then 64 bytes of 4-bit indices, element j in bits
 * 4 * (j % 2) of byte 4 + j / 2.
 *
 * Nothing here is tuned: one key at a time, its 128 K and V centroids decoded into two
 * small arrays, then g dot products and g scaled adds.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define HD 128
#define ROW 68
#define MAX_G 64

/* One (batch, KV head) unit: g queries q [g][128] (unrotated), L keys and values. */
static void decode_unit(const float *q, int g, const uint8_t *K, const uint8_t *V, int L,
                        const float *rk, const float *rv, const float *ck, const float *cv,
                        float scale, float *out) {
  float qr[MAX_G][HD], acc[MAX_G][HD], m[MAX_G], l[MAX_G];
  float kd[HD], vd[HD];
  for (int h = 0; h < g; ++h) {
    for (int i = 0; i < HD; ++i) {
      float s = 0.f;
      for (int j = 0; j < HD; ++j) s += rk[i * HD + j] * q[h * HD + j];
      qr[h][i] = s * scale;
      acc[h][i] = 0.f;
    }
    m[h] = -INFINITY;
    l[h] = 0.f;
  }
  for (int t = 0; t < L; ++t) {
    const uint8_t *kr = K + (size_t)t * ROW, *vr = V + (size_t)t * ROW;
    float nk, nv;
    memcpy(&nk, kr, 4);
    memcpy(&nv, vr, 4);
    for (int j = 0; j < HD; ++j) {
      kd[j] = ck[(kr[4 + j / 2] >> (4 * (j % 2))) & 15];
      vd[j] = nv * cv[(vr[4 + j / 2] >> (4 * (j % 2))) & 15];
    }
    for (int h = 0; h < g; ++h) {
      float s = 0.f;
      for (int j = 0; j < HD; ++j) s += qr[h][j] * kd[j];
      s *= nk;
      if (s > m[h]) {
        const float a = (m[h] == -INFINITY) ? 0.f : expf(m[h] - s);
        l[h] *= a;
        for (int j = 0; j < HD; ++j) acc[h][j] *= a;
        m[h] = s;
      }
      const float p = expf(s - m[h]);
      l[h] += p;
      for (int j = 0; j < HD; ++j) acc[h][j] += p * vd[j];
    }
  }
  for (int h = 0; h < g; ++h)
    for (int i = 0; i < HD; ++i) {
      float s = 0.f;
      for (int j = 0; j < HD; ++j) s += rv[j * HD + i] * acc[h][j];  /* (R^T a)_i = sum_j R[j][i] a_j */
      out[h * HD + i] = s / l[h];
    }
}

/*
 * q [B][Hq][128] fp32; k_cache, v_cache [B][Hkv][L] turbo4 rows; rk, rv the key and value
 * rotations R (fp32 [128][128] row-major, y = R u); ck, cv the 16 fp32 centroids; scale
 * the softmax scale; out [B][Hq][128] fp32.  Query head h reads KV head h / (Hq / Hkv).
 * threads: OpenMP threads over the B * Hkv units (1 = a single core).  Returns the
 * number of threads used, or -1 on bad arguments.
 */
int tq_cpu_decode_turbo4(const float *q, const uint8_t *k_cache, const uint8_t *v_cache, int B,
                         int Hq, int Hkv, int L, const float *rk, const float *rv, const float *ck,
                         const float *cv, float scale, float *out, int threads) {
  if (B < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq / Hkv > MAX_G || L < 1 || threads < 1) return -1;
  const int g = Hq / Hkv, units = B * Hkv;
  int used = 1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
  for (int u = 0; u < units; ++u) {
    const int b = u / Hkv, kvh = u % Hkv;
    const size_t off = (size_t)u * L * ROW;
    decode_unit(q + ((size_t)b * Hq + (size_t)kvh * g) * HD, g, k_cache + off, v_cache + off, L, rk, rv,
                ck, cv, scale, out + ((size_t)b * Hq + (size_t)kvh * g) * HD);
#ifdef _OPENMP
    if (u == 0) used = omp_get_num_threads();
#endif
  }
  return used;
}
