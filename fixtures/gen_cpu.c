/* Host implementation of the fixture generator of fixtures/__init__.py
 * (SplitMix64 words, Box-Muller normals in double, rounded to float and,
 * for bf16 models, to bfloat16 with round-to-nearest-even), parallel over
 * elements with OpenMP. Used for the oracle's full-size weights. */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline double std_normal(uint64_t key, uint64_t i) {
  const uint64_t a = mix64(key + (2 * i + 1) * GAMMA);
  const uint64_t b = mix64(key + (2 * i + 2) * GAMMA);
  const double u1 = (double)((a >> 11) + 1) * (1.0 / 9007199254740992.0);
  const double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

static inline float round_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u = (u + (((u >> 16) & 1u) + 0x7FFFu)) & 0xFFFF0000u;
  memcpy(&f, &u, 4);
  return f;
}

void fx_fill_normal_host(float* out, int64_t count, int64_t start, uint64_t key, double sd, uint64_t nkey,
                         double nsd, int noise, int bf16) {
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < count; ++e) {
    const uint64_t i = (uint64_t)(start + e);
    double v = sd * std_normal(key, i);
    if (noise) v = v + nsd * std_normal(nkey, i);
    float f = (float)v;
    out[e] = bf16 ? round_bf16(f) : f;
  }
}
