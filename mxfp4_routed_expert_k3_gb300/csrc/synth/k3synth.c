/*
 * k3synth.c -- seeded, counter-based synthetic input generator.
 *
 * This module only draws random numbers.  It holds none of the layer's
 * arithmetic (no routing, no MXFP4 decoding, no activation); both the CUDA
 * path's tests/benchmark and the CPU oracle take their inputs from here, so
 * the two sides see identical bytes.
 *
 * Every value is a pure function of (seed, stream, index): element i of a
 * tensor is derived from splitmix64 applied to a key built from the three
 * numbers, so results do not depend on thread count or on the order in
 * which elements are produced.  Normal deviates use the Box-Muller transform
 * with a logarithm and a cosine written here from their series, using only
 * IEEE +,-,*,/ and sqrt (compile with -ffp-contract=off), so x86-64 and
 * aarch64 hosts produce the same bits.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* splitmix64 finaliser (Steele, Lea, Flood 2014). */
static inline uint64_t k3s_mix(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t k3s_counter_u64(uint64_t seed, uint64_t stream, uint64_t index) {
  uint64_t k = k3s_mix(seed ^ 0x5851F42D4C957F2Dull);
  k = k3s_mix(k ^ (stream * 0xD1B54A32D192ED03ull));
  return k3s_mix(k + index);
}

/* natural log for x in (0, 1]: x = m * 2^e with m in [sqrt(1/2), sqrt(2)),
 * ln m = 2 * atanh(t), t = (m-1)/(m+1), |t| < 0.172, series to t^25. */
static double k3s_log(double x) {
  int e;
  double m = frexp(x, &e);
  if (m < 0.70710678118654752440) {
    m *= 2.0;
    e -= 1;
  }
  double t = (m - 1.0) / (m + 1.0);
  double t2 = t * t, term = t, sum = 0.0;
  for (int k = 1; k <= 25; k += 2) {
    sum += term / (double)k;
    term *= t2;
  }
  return 2.0 * sum + (double)e * 0.69314718055994530942;
}

/* cos(2*pi*v) for v in [0, 1): fold to r in [0, 1/4] turns, Taylor to x^24. */
static double k3s_cos_turns(double v) {
  double r = v - floor(v + 0.5); /* [-1/2, 1/2] */
  if (r < 0) r = -r;             /* cos is even */
  double sign = 1.0;
  if (r > 0.25) {                /* cos(2pi r) = -cos(2pi (1/2 - r)) */
    r = 0.5 - r;
    sign = -1.0;
  }
  double a = 6.28318530717958647692 * r; /* [0, pi/2] */
  double a2 = a * a, term = 1.0, sum = 0.0;
  for (int k = 0; k <= 12; ++k) {
    sum += term;
    term *= -a2 / (double)((2 * k + 1) * (2 * k + 2));
  }
  return sign * sum;
}

/* double -> bf16 bits, round to nearest even on the float value. */
static uint16_t k3s_bf16_bits(double v) {
  float f = (float)v;
  union { float f; uint32_t u; } c;
  c.f = f;
  uint32_t u = c.u;
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFF) ? 0x40 : 0));
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static double k3s_unit_open(uint64_t h) { /* (0, 1] */
  return ((double)(h >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}
static double k3s_unit(uint64_t h) { /* [0, 1) */
  return (double)(h >> 11) * (1.0 / 9007199254740992.0);
}

double k3s_normal(uint64_t seed, uint64_t stream, uint64_t index) {
  double u1 = k3s_unit_open(k3s_counter_u64(seed, stream, 2 * index));
  double u2 = k3s_unit(k3s_counter_u64(seed, stream, 2 * index + 1));
  return sqrt(-2.0 * k3s_log(u1)) * k3s_cos_turns(u2);
}

/* out[i] = bf16(mean + std * N(0,1)) for element (index0 + i) of the stream. */
void k3s_fill_bf16_normal(uint64_t seed, uint64_t stream, uint64_t index0,
                          double mean, double std, uint16_t* out, size_t n) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i)
    out[i] = k3s_bf16_bits(mean + std * k3s_normal(seed, stream, index0 + (uint64_t)i));
}

/* out[i] = lo + (hi - lo) * U[0,1), rounded to float. */
void k3s_fill_f32_uniform(uint64_t seed, uint64_t stream, uint64_t index0,
                          double lo, double hi, float* out, size_t n) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i)
    out[i] = (float)(lo + (hi - lo) * k3s_unit(k3s_counter_u64(seed, stream, index0 + (uint64_t)i)));
}

/* Uniform bytes over the full range 0..255: byte i is byte (i % 8) of the
 * counter value for index i / 8. */
void k3s_fill_u8_full(uint64_t seed, uint64_t stream, uint8_t* out, size_t n) {
  size_t words = n / 8;
#pragma omp parallel for schedule(static)
  for (long long w = 0; w < (long long)words; ++w) {
    uint64_t h = k3s_counter_u64(seed, stream, (uint64_t)w);
    for (int b = 0; b < 8; ++b) out[(size_t)w * 8 + b] = (uint8_t)(h >> (8 * b));
  }
  if (words * 8 < n) {
    uint64_t h = k3s_counter_u64(seed, stream, (uint64_t)words);
    for (size_t i = words * 8; i < n; ++i) out[i] = (uint8_t)(h >> (8 * (i - words * 8)));
  }
}

/* Uniform integers in [lo, hi] (inclusive), one counter value per element. */
void k3s_fill_u8_range(uint64_t seed, uint64_t stream, uint8_t lo, uint8_t hi,
                       uint8_t* out, size_t n) {
  uint64_t span = (uint64_t)hi - (uint64_t)lo + 1u;
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i)
    out[i] = (uint8_t)(lo + k3s_counter_u64(seed, stream, (uint64_t)i) % span);
}

/* A seeded permutation of 0..n-1 (Fisher-Yates driven by the counter). */
void k3s_permutation(uint64_t seed, uint64_t stream, int32_t* out, int n) {
  for (int i = 0; i < n; ++i) out[i] = i;
  for (int i = n - 1; i > 0; --i) {
    uint64_t j = k3s_counter_u64(seed, stream, (uint64_t)i) % (uint64_t)(i + 1);
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}

int k3s_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
