// Host-side construction of codebooks, rotations and the QJL matrix (fp64), and
// the fp16 operand tables used by the tensor-core decode.
//
// Codebooks follow "turboquant_plus: how the turbo4 KV format came back",
// section 5 (16-level table for N(0, 1/d), d = 128: conditional means of the
// quantile cells) and sections 5 and 9 (Lloyd-Max on the Gaussian).  The dense
// rotation is the Q factor of a seeded Gaussian ("TurboQuant fused Triton
// kernels deep dive", trick 1); the QJL matrix is a second, independent
// Gaussian (trick 2; post-mortem section 10 on independent seeds).
#include <cuda_fp16.h>

#include <cmath>
#include <map>
#include <mutex>
#include <tuple>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "tq_internal.h"

namespace tq {

namespace {

thread_local char g_last_error[512] = "";

const double kSqrt2 = 1.4142135623730950488;
const double kPi = 3.14159265358979323846;

double std_pdf(double x) {
  if (std::isinf(x)) return 0.0;
  return std::exp(-0.5 * x * x) / std::sqrt(2.0 * kPi);
}

double std_cdf(double x) { return 0.5 * std::erfc(-x / kSqrt2); }

// P(a < Z < b), evaluated on the tail side that avoids cancellation.
double std_mass(double a, double b) {
  if (a >= 0.0) return 0.5 * (std::erfc(a / kSqrt2) - std::erfc(b / kSqrt2));
  if (b <= 0.0) return 0.5 * (std::erfc(-b / kSqrt2) - std::erfc(-a / kSqrt2));
  return 1.0 - 0.5 * std::erfc(-a / kSqrt2) - 0.5 * std::erfc(b / kSqrt2);
}

double std_quantile(double p) {
  if (p <= 0.0) return -INFINITY;
  if (p >= 1.0) return INFINITY;
  double lo = -40.0, hi = 40.0;
  while (hi - lo > 1e-15) {
    double mid = 0.5 * (lo + hi);
    if (mid == lo || mid == hi) break;
    if (std_cdf(mid) < p)
      lo = mid;
    else
      hi = mid;
  }
  return 0.5 * (lo + hi);
}

double cond_mean(double a, double b) { return (std_pdf(a) - std_pdf(b)) / std_mass(a, b); }

// Regularized incomplete beta I_x(a, b) for x <= (a + 1) / (a + b + 2), by the continued
// fraction of DLMF 8.17.22 evaluated with the modified Lentz method.
double betainc_cf(double a, double b, double x) {
  if (x <= 0.0) return 0.0;
  const double log_front = a * std::log(x) + b * std::log1p(-x) - std::log(a) -
                           (std::lgamma(a) + std::lgamma(b) - std::lgamma(a + b));
  const double tiny = 1e-300;
  double f = 1.0, c = 1.0, dd = 0.0;
  for (int i = 0; i <= 2000; ++i) {
    double num;  // the i-th numerator d_i of 1 / (1 + d_1 / (1 + d_2 / ...))
    if (i == 0) {
      num = 1.0;
    } else {
      const int m = i / 2;
      num = (i % 2 == 0) ? m * (b - m) * x / ((a + 2.0 * m - 1.0) * (a + 2.0 * m))
                         : -(a + m) * (a + b + m) * x / ((a + 2.0 * m) * (a + 2.0 * m + 1.0));
    }
    dd = 1.0 + num * dd;
    if (std::fabs(dd) < tiny) dd = tiny;
    dd = 1.0 / dd;
    c = 1.0 + num / c;
    if (std::fabs(c) < tiny) c = tiny;
    const double delta = c * dd;
    f *= delta;
    if (std::fabs(delta - 1.0) < 1e-16) break;
  }
  return std::exp(log_front) * (f - 1.0);
}

// I_t(al, al) for the symmetric case, with the fraction on the side where it converges.
double betainc_sym(double al, double t) {
  if (t <= 0.0) return 0.0;
  if (t >= 1.0) return 1.0;
  return t <= 0.5 ? betainc_cf(al, al, t) : 1.0 - betainc_cf(al, al, 1.0 - t);
}

// Law of one coordinate X of a uniform point on the unit sphere in R^d: density
// proportional to (1 - x^2)^m on [-1, 1], m = (d - 3)/2, i.e. (1 + X)/2 ~ Beta(al, al),
// al = m + 1.  P(a < X < b), taken on the side that avoids cancellation.
double sphere_mass(double al, double a, double b) {
  const double ta = a <= -1.0 ? 0.0 : (a >= 1.0 ? 1.0 : 0.5 * (1.0 + a));
  const double tb = b <= -1.0 ? 0.0 : (b >= 1.0 ? 1.0 : 0.5 * (1.0 + b));
  if (tb <= 0.5) return betainc_sym(al, tb) - betainc_sym(al, ta);
  if (ta >= 0.5) return betainc_sym(al, 1.0 - ta) - betainc_sym(al, 1.0 - tb);
  return 1.0 - betainc_sym(al, ta) - betainc_sym(al, 1.0 - tb);
}

// E[X | a < X < b]: the first moment integrates in closed form,
// int x (1 - x^2)^m dx = -(1 - x^2)^al / (2 al), over Z = 2 4^m B(al, al).
double sphere_cond_mean(double al, double a, double b) {
  const double m = al - 1.0;
  const double log_z = std::log(2.0) + m * std::log(4.0) + 2.0 * std::lgamma(al) - std::lgamma(2.0 * al);
  const double ga = (a > -1.0 && a < 1.0) ? std::pow(1.0 - a * a, al) : 0.0;
  const double gb = (b > -1.0 && b < 1.0) ? std::pow(1.0 - b * b, al) : 0.0;
  return (ga - gb) / (2.0 * al) * std::exp(-log_z) / sphere_mass(al, a, b);
}

}  // namespace

cudaError_t kernel_smem_attr(const void *func, int bytes, bool max_shared) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::map<std::tuple<const void *, int, int, bool>, bool> done;
  const auto key = std::make_tuple(func, dev, bytes, max_shared);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count(key)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && max_shared)
    e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) done[key] = true;
  return e;
}

cudaError_t kernel_occupancy(const void *func, int threads, size_t smem, int *blocks) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::map<std::tuple<const void *, int, int, size_t>, int> known;
  const auto key = std::make_tuple(func, dev, threads, smem);
  std::lock_guard<std::mutex> lock(mu);
  const auto it = known.find(key);
  if (it != known.end()) {
    *blocks = it->second;
    return cudaSuccess;
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, func, threads, smem);
  if (e == cudaSuccess) known[key] = *blocks;
  return e;
}

void set_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
}

const char *last_error() { return g_last_error; }

bool make_codebook_f64(int bits, int d, int kind, double *c) {
  const int K = 1 << bits;
  const double sigma = 1.0 / std::sqrt((double)d);
  std::vector<double> t(K + 1), cs(K);
  for (int k = 0; k <= K; ++k) t[k] = std_quantile((double)k / K);
  for (int k = 0; k < K; ++k) cs[k] = cond_mean(t[k], t[k + 1]);  // QUANTILE, standard units
  if (kind == TQ_CB_SPHERE) {
    // Lloyd-Max under the sphere marginal, from the Gaussian QUANTILE start (in x units)
    const double al = 0.5 * (d - 1);
    std::vector<double> cx(K), cn(K);
    for (int k = 0; k < K; ++k) cx[k] = cs[k] * sigma;
    for (int it = 0; it < 1000000; ++it) {
      double moved = 0.0;
      for (int k = 0; k < K; ++k) {
        const double a = k == 0 ? -1.0 : 0.5 * (cx[k - 1] + cx[k]);
        const double b = k == K - 1 ? 1.0 : 0.5 * (cx[k] + cx[k + 1]);
        cn[k] = sphere_cond_mean(al, a, b);
        moved = std::fmax(moved, std::fabs(cn[k] - cx[k]));
      }
      cx = cn;
      if (moved < 1e-13) break;
    }
    for (int k = 0; k < K; ++k) c[k] = cx[k];
    return true;
  }
  if (kind == TQ_CB_LLOYD) {
    std::vector<double> cn(K);
    for (int it = 0; it < 1000000; ++it) {
      t[0] = -INFINITY;
      t[K] = INFINITY;
      for (int k = 1; k < K; ++k) t[k] = 0.5 * (cs[k - 1] + cs[k]);
      double moved = 0.0;
      for (int k = 0; k < K; ++k) {
        cn[k] = cond_mean(t[k], t[k + 1]);
        moved = std::fmax(moved, std::fabs(cn[k] - cs[k]));
      }
      cs = cn;
      if (moved * sigma < 1e-13) break;
    }
  } else if (kind != TQ_CB_QUANTILE) {
    return false;
  }
  for (int k = 0; k < K; ++k) c[k] = cs[k] * sigma;
  return true;
}

void store_codebook(const double *c64, int K, float *c32, float *b32) {
  for (int k = 0; k < K; ++k) c32[k] = (float)c64[k];
  if (b32)
    for (int k = 0; k + 1 < K; ++k) b32[k] = (float)(((double)c32[k] + (double)c32[k + 1]) / 2.0);
}

void splitmix64_fill(uint64_t seed, uint64_t *out, size_t n) {
  uint64_t state = seed;
  for (size_t i = 0; i < n; ++i) {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    out[i] = z ^ (z >> 31);
  }
}

void gaussian_fill(uint64_t seed, double *out, size_t n) {
  const size_t pairs = (n + 1) / 2;
  std::vector<uint64_t> raw(2 * pairs);
  splitmix64_fill(seed, raw.data(), raw.size());
  for (size_t p = 0; p < pairs; ++p) {
    const double u1 = (double)((raw[2 * p] >> 11) + 1) * 0x1.0p-53;
    const double u2 = (double)(raw[2 * p + 1] >> 11) * 0x1.0p-53;
    const double r = std::sqrt(-2.0 * std::log(u1));
    out[2 * p] = r * std::cos(2.0 * kPi * u2);
    if (2 * p + 1 < n) out[2 * p + 1] = r * std::sin(2.0 * kPi * u2);
  }
}

// Householder QR of the seeded Gaussian G (row-major d x d); returns Q with the
// signs fixed so that diag(R) > 0, which makes the factorisation unique.
bool dense_rotation_f64(uint64_t seed, int d, double *pi) {
  std::vector<double> A((size_t)d * d);
  gaussian_fill(seed, A.data(), A.size());
  std::vector<double> V((size_t)d * d, 0.0);  // Householder vectors, column k in V[:, k]
  std::vector<double> rdiag(d);
  for (int k = 0; k < d; ++k) {
    double nrm = 0.0;
    for (int i = k; i < d; ++i) nrm += A[(size_t)i * d + k] * A[(size_t)i * d + k];
    nrm = std::sqrt(nrm);
    if (nrm == 0.0) return false;
    const double x0 = A[(size_t)k * d + k];
    const double alpha = x0 >= 0.0 ? -nrm : nrm;  // reflect x onto alpha e_k
    double vnorm2 = 0.0;
    for (int i = k; i < d; ++i) {
      double v = A[(size_t)i * d + k] - (i == k ? alpha : 0.0);
      V[(size_t)i * d + k] = v;
      vnorm2 += v * v;
    }
    const double inv = 1.0 / std::sqrt(vnorm2);
    for (int i = k; i < d; ++i) V[(size_t)i * d + k] *= inv;
    for (int j = k; j < d; ++j) {  // A[k:, j] -= 2 v (v . A[k:, j])
      double dot = 0.0;
      for (int i = k; i < d; ++i) dot += V[(size_t)i * d + k] * A[(size_t)i * d + j];
      for (int i = k; i < d; ++i) A[(size_t)i * d + j] -= 2.0 * V[(size_t)i * d + k] * dot;
    }
    rdiag[k] = A[(size_t)k * d + k];
  }
  // Q = H_0 H_1 ... H_{d-1} I
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) pi[(size_t)i * d + j] = (i == j) ? 1.0 : 0.0;
  for (int k = d - 1; k >= 0; --k) {
    for (int j = 0; j < d; ++j) {
      double dot = 0.0;
      for (int i = k; i < d; ++i) dot += V[(size_t)i * d + k] * pi[(size_t)i * d + j];
      for (int i = k; i < d; ++i) pi[(size_t)i * d + j] -= 2.0 * V[(size_t)i * d + k] * dot;
    }
  }
  for (int j = 0; j < d; ++j)
    if (rdiag[j] < 0.0)
      for (int i = 0; i < d; ++i) pi[(size_t)i * d + j] = -pi[(size_t)i * d + j];
  return true;
}

F16Table make_f16_table(const float *c32, int K) {
  // Magnitudes of the symmetric codebook, largest first: mag[m] = |c_m|, m < K/2.
  F16Table t;
  const int nm = K / 2;
  double mag[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int m = 0; m < nm; ++m) mag[m] = std::fabs((double)c32[m]);
  double best_err = 1e30, best_a = 1.0;
  for (int s = 0; s < 65536; ++s) {
    const double a = 1.0 + s / 65536.0;
    double err = 0.0;
    for (int m = 0; m < nm; ++m) {
      const double v = a * mag[m];
      const double h = (double)__half2float(__float2half_rn((float)v));
      err = std::fmax(err, std::fabs(h - v) / v);
    }
    if (err < best_err) {
      best_err = err;
      best_a = a;
    }
  }
  uint8_t lo[8] = {0}, hi[8] = {0};
  for (int m = 0; m < nm; ++m) {
    __half h = __float2half_rn((float)(best_a * mag[m]));
    uint16_t bits;
    std::memcpy(&bits, &h, 2);
    lo[m] = (uint8_t)(bits & 0xFF);
    hi[m] = (uint8_t)(bits >> 8);
  }
  std::memcpy(t.lo, lo, 8);
  std::memcpy(t.hi, hi, 8);
  // signed entries in index order: idx < K/2 is -mag[idx], idx >= K/2 is +mag[K-1-idx]
  for (int idx = 0; idx < K; ++idx) {
    const int m = idx < nm ? idx : K - 1 - idx;
    const uint16_t bits = (uint16_t)(lo[m] | (hi[m] << 8) | (idx < nm ? 0x8000 : 0));
    t.c16[idx / 2] |= (uint32_t)bits << (16 * (idx % 2));
  }
  t.alpha = (float)best_a;
  t.max_rel_err = (float)best_err;
  return t;
}

BucketTable make_bucket_table(const float *b, int nb) {
  BucketTable t;
  if (nb < 1) return t;
  double gap = 1e300;
  for (int k = 0; k + 1 < nb; ++k) gap = std::fmin(gap, (double)b[k + 1] - (double)b[k]);
  if (nb == 1) gap = 1.0;
  if (!(gap > 0.0) || !std::isfinite(gap)) return t;
  const double w = 0.4 * gap, lo = (double)b[0] - w, delta = 0.05 * w;
  const int n = (int)std::ceil(((double)b[nb - 1] - lo) / w) + 2;
  if (n > GRID_CELLS) return t;
  for (int c = 0; c < n; ++c) {
    const double a = lo + c * w - delta, z = lo + (c + 1) * w + delta;
    int cnt = 0, listed = 0;
    float e = INFINITY;
    for (int k = 0; k < nb; ++k) {
      if ((double)b[k] < a) {
        ++cnt;
      } else if ((double)b[k] <= z) {
        if (listed == 1) return BucketTable{};
        e = b[k];
        ++listed;
      }
    }
    t.cnt[c] = (uint8_t)cnt;
    t.e[c] = e;
  }
  t.scale = (float)(1.0 / w);
  t.offset = (float)(-lo / w);
  t.n = n;
  return t;
}

}  // namespace tq
