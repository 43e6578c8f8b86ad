/*
 * Seeded synthetic-input generator shared by the oracle side and the CUDA side
 * of the tests and the benchmark.  It holds none of the MoE layer's arithmetic:
 * it only turns (seed, tensor id, element index) into a number.
 *
 * Every element is addressable on its own (a counter-based hash, no sequential
 * state), so a slice of a large tensor -- one expert's weight matrix, a few
 * token rows -- can be generated without generating the rest, and the result
 * does not depend on the number of threads.
 *
 *   u64 key   = mix64(seed * 0x9E3779B97F4A7C15 ^ mix64(tensor_id + 0x632BE59BD9B4E019))
 *   u1, u2    = (mix64(key + 2i) >> 11 + 1) * 2^-53,  (mix64(key + 2i + 1) >> 11) * 2^-53
 *   z         = sqrt(-2 ln u1) * cos(2 pi u2)            (Box-Muller, one normal per element)
 *   value     = mean + sigma * z, rounded once to the storage type (bf16: round to nearest even)
 *
 * mix64 is the SplitMix64 finaliser (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t tensor_key(uint64_t seed, uint64_t tensor_id) {
  return mix64(seed * 0x9E3779B97F4A7C15ULL ^ mix64(tensor_id + 0x632BE59BD9B4E019ULL));
}

static inline double normal_at(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  double u1 = (double)((mix64(key + 2 * i) >> 11) + 1) * 0x1.0p-53; /* (0, 1] */
  double u2 = (double)(mix64(key + 2 * i + 1) >> 11) * 0x1.0p-53;   /* [0, 1) */
  return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

static inline double uniform_at(uint64_t key, uint64_t i) {
  return (double)(mix64(key + i) >> 11) * 0x1.0p-53; /* [0, 1) */
}

/* double -> bf16 bits with a single round-to-nearest-even: round to float with
 * round-to-odd first (exact for the later 8-bit rounding), then RNE to bf16. */
static inline uint16_t bf16_from_double(double d) {
  float f = (float)d;
  if ((double)f != d) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 1u) == 0u) f = nextafterf(f, (float)(d > (double)f ? INFINITY : -INFINITY));
  }
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void wl_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t offset, int64_t n,
                    double mean, double sigma, uint16_t *out) {
  const uint64_t key = tensor_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = bf16_from_double(mean + sigma * normal_at(key, offset + (uint64_t)i));
}

void wl_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t offset, int64_t n,
                   double mean, double sigma, float *out) {
  const uint64_t key = tensor_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = (float)(mean + sigma * normal_at(key, offset + (uint64_t)i));
}

void wl_uniform_f64(uint64_t seed, uint64_t tensor_id, uint64_t offset, int64_t n, double *out) {
  const uint64_t key = tensor_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = uniform_at(key, offset + (uint64_t)i);
}

/* A seeded permutation of 0..n-1 (Fisher-Yates driven by the same hash). */
void wl_permutation(uint64_t seed, uint64_t tensor_id, int64_t n, int32_t *out) {
  const uint64_t key = tensor_key(seed, tensor_id);
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  for (int64_t i = n - 1; i > 0; --i) {
    int64_t j = (int64_t)(mix64(key + (uint64_t)i) % (uint64_t)(i + 1));
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}

/* Uniform integers in [0, m) (used for synthetic routing tables in isolated stage tests). */
void wl_randint(uint64_t seed, uint64_t tensor_id, uint64_t offset, int64_t n, int64_t m, int32_t *out) {
  const uint64_t key = tensor_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(mix64(key + offset + (uint64_t)i) % (uint64_t)m);
}
