/*
 * Counter-based generator for the synthetic inputs of the MoE layer.
 *
 * Every element is a pure function of (seed, stream, index), so any slice of
 * any tensor can be regenerated independently (per expert, per token) on the
 * host without holding the whole tensor.  This file holds no arithmetic of the
 * MoE method itself: it only draws numbers.
 *
 * Definition (fixed; changing it changes every synthetic input):
 *   splitmix64(x): x += 0x9E3779B97F4A7C15; x = (x ^ x>>30) * 0xBF58476D1CE4E5B9;
 *                  x = (x ^ x>>27) * 0x94D049BB133111EB; return x ^ x>>31
 *   base(seed, stream) = splitmix64(seed ^ splitmix64(stream * 0xD1B54A32D192ED03 + 1))
 *   normal element i:  q = i>>1, r1 = splitmix64(base + 2q), r2 = splitmix64(base + 2q + 1)
 *                      u1 = ((r1>>11) + 1) * 2^-53 in (0,1],  u2 = (r2>>11) * 2^-53 in [0,1)
 *                      rho = sqrt(-2 ln u1), phi = 2 pi u2
 *                      z = rho cos(phi) for even i, rho sin(phi) for odd i   (Box-Muller)
 *                      value = (float)(mean + std * z), then rounded to bf16 (nearest-even)
 *   integer element i: value = lo + splitmix64(base + i) mod (hi - lo + 1)
 *   uniform element i: u = (splitmix64(base + i) >> 11) * 2^-53 in [0,1)
 */
#include <math.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static inline uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

static inline uint64_t stream_base(uint64_t seed, uint64_t stream) {
  return splitmix64(seed ^ splitmix64(stream * 0xD1B54A32D192ED03ull + 1ull));
}

/* float -> bf16 bits, round to nearest even; NaN kept quiet. */
static inline uint16_t f32_to_bf16(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  if ((v.u & 0x7F800000u) == 0x7F800000u && (v.u & 0x007FFFFFu)) return (uint16_t)((v.u >> 16) | 0x40u);
  uint32_t lsb = (v.u >> 16) & 1u;
  v.u += 0x7FFFu + lsb;
  return (uint16_t)(v.u >> 16);
}

static inline double normal_at(uint64_t base, int64_t i) {
  const double two_m53 = 1.0 / 9007199254740992.0;
  uint64_t q = (uint64_t)i >> 1;
  uint64_t r1 = splitmix64(base + 2u * q);
  uint64_t r2 = splitmix64(base + 2u * q + 1u);
  double u1 = (double)((r1 >> 11) + 1u) * two_m53;
  double u2 = (double)(r2 >> 11) * two_m53;
  double rho = sqrt(-2.0 * log(u1));
  double phi = 6.283185307179586 * u2;
  return (i & 1) ? rho * sin(phi) : rho * cos(phi);
}

void synth_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t stream, int64_t offset,
                       double mean, double stdev) {
  uint64_t base = stream_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float v = (float)(mean + stdev * normal_at(base, offset + i));
    out[i] = f32_to_bf16(v);
  }
}

void synth_normal_f32(float* out, int64_t n, uint64_t seed, uint64_t stream, int64_t offset,
                      double mean, double stdev) {
  uint64_t base = stream_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(mean + stdev * normal_at(base, offset + i));
}

void synth_int_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t stream, int64_t offset,
                    int32_t lo, int32_t hi) {
  uint64_t base = stream_base(seed, stream);
  uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo + 1);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    int64_t v = (int64_t)lo + (int64_t)(splitmix64(base + (uint64_t)(offset + i)) % span);
    out[i] = f32_to_bf16((float)v);
  }
}

void synth_uniform_f64(double* out, int64_t n, uint64_t seed, uint64_t stream, int64_t offset) {
  const double two_m53 = 1.0 / 9007199254740992.0;
  uint64_t base = stream_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (double)(splitmix64(base + (uint64_t)(offset + i)) >> 11) * two_m53;
}

int synth_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
