/*
 * Seeded synthetic inputs for the FC-layer GEMMs (bf16 bit patterns).
 *
 * This file holds no part of the method's arithmetic: it only draws the
 * numbers that both the fp64 oracle and the GPU path consume.  Every element
 * is a pure function of (seed, tensor id, element index), so any sub-range can
 * be regenerated independently and in parallel.
 *
 * Definition (counter-based SplitMix64, Steele/Lea/Flood 2014, with the
 * finaliser constants published in Vigna's reference implementation):
 *   gamma        = 0x9E3779B97F4A7C15
 *   mix(z)       = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *                  z ^= z >> 27; z *= 0x94D049BB133111EB; z ^ (z >> 31)
 *   x0           = seed * 2^32 + tid * 2^16            (mod 2^64)
 *   draw(k)      = mix(x0 + (k + 1) * gamma)           (mod 2^64)
 * This is exactly the k-th output of a SplitMix64 generator seeded with x0.
 *
 * Normal element n (Box-Muller, one value per pair of draws):
 *   u1 = ((draw(2n)   >> 11) + 0.5) * 2^-53     in (0, 1)
 *   u2 =  (draw(2n+1) >> 11)        * 2^-53     in [0, 1)
 *   v  = mean + sigma * sqrt(-2 ln u1) * cos(2 pi u2)      (double)
 *   bits = bf16_rne(float_rne(v))
 * Ternary element n: (draw(n) mod 3) - 1, exactly representable in bf16.
 * Small-integer element n: (draw(n) mod (2h+1)) - h.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_base(uint64_t seed, uint64_t tid) {
  return (seed << 32) + (tid << 16);
}

static inline uint64_t draw(uint64_t x0, uint64_t k) {
  return mix64(x0 + (k + 1ULL) * GAMMA);
}

/* float32 -> bf16 bits, round to nearest even (inputs here are finite). */
static inline uint16_t f32_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void fc_inputs_splitmix64(uint64_t x0, int64_t count, uint64_t* out) {
  for (int64_t k = 0; k < count; ++k) out[k] = draw(x0, (uint64_t)k);
}

void fc_inputs_normal_bf16(uint64_t seed, uint64_t tid, int64_t start,
                           int64_t count, double mean, double sigma,
                           uint16_t* out) {
  const uint64_t x0 = stream_base(seed, tid);
  const double two_pi = 6.283185307179586476925286766559;
  const double inv53 = 1.0 / 9007199254740992.0; /* 2^-53 */
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    const uint64_t n = (uint64_t)(start + i);
    const double u1 = ((double)(draw(x0, 2 * n) >> 11) + 0.5) * inv53;
    const double u2 = (double)(draw(x0, 2 * n + 1) >> 11) * inv53;
    const double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
    out[i] = f32_to_bf16_bits((float)(mean + sigma * z));
  }
}

void fc_inputs_small_int_bf16(uint64_t seed, uint64_t tid, int64_t start,
                              int64_t count, int64_t h, uint16_t* out) {
  const uint64_t x0 = stream_base(seed, tid);
  const uint64_t span = (uint64_t)(2 * h + 1);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    const uint64_t n = (uint64_t)(start + i);
    const int64_t v = (int64_t)(draw(x0, n) % span) - h;
    out[i] = f32_to_bf16_bits((float)v);
  }
}
