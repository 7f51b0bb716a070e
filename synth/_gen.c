/* Seeded input generation helpers for synth/__init__.py: counter-based
 * splitmix64 (Steele, Lea & Flood, OOPSLA 2014) and Box-Muller normals.
 * Output i of a stream with state s is mix(s + (i + 1) * gamma). */
#include <math.h>
#include <stdint.h>

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline double unif(uint64_t state, int64_t i) {
  uint64_t z = mix64(state + (uint64_t)(i + 1) * 0x9E3779B97F4A7C15ULL);
  return ((double)(z >> 11) + 1.0) * 0x1.0p-53;
}

/* out[i] = mean + std * normal_i, i < n, as float32; normals come in
 * Box-Muller pairs from uniforms (2m, 2m+1). */
void synth_normals_f32(uint64_t state, int64_t n, double mean, double std, float* out) {
  const double two_pi = 6.283185307179586476925286766559;
  int64_t m = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < m; ++p) {
    double r = sqrt(-2.0 * log(unif(state, 2 * p)));
    double a = two_pi * unif(state, 2 * p + 1);
    out[2 * p] = (float)(mean + std * (r * cos(a)));
    if (2 * p + 1 < n) out[2 * p + 1] = (float)(mean + std * (r * sin(a)));
  }
}

/* out[i] = (float)(base[i] + std * normal_i), base in float64. */
void synth_add_normals_f32(uint64_t state, int64_t n, double std, const double* base, float* out) {
  const double two_pi = 6.283185307179586476925286766559;
  int64_t m = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < m; ++p) {
    double r = sqrt(-2.0 * log(unif(state, 2 * p)));
    double a = two_pi * unif(state, 2 * p + 1);
    out[2 * p] = (float)(base[2 * p] + std * (r * cos(a)));
    if (2 * p + 1 < n) out[2 * p + 1] = (float)(base[2 * p + 1] + std * (r * sin(a)));
  }
}

/* Round float32 to the nearest bf16 value in place (ties to even). */
void synth_round_bf16(int64_t n, float* x) {
  uint32_t* b = (uint32_t*)x;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint32_t v = b[i];
    v = (v + 0x7FFFu + ((v >> 16) & 1u)) & 0xFFFF0000u;
    b[i] = v;
  }
}
