/*
 * Seeded synthetic inputs for the batch-1 decode workloads.
 *
 * This file holds no part of the decoder's arithmetic: it only draws random numbers and rounds them
 * to IEEE binary16, so that the CPU oracle and the GPU library can be fed the very same bytes.
 *
 * Generator (the pages fix none, so this one is chosen and documented):
 *   - SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014),
 *     used counter-style: draw i of a stream is mix64(base + (i + 1) * GOLDEN), where base is derived from
 *     (seed, tensor_id). Any element can therefore be drawn on its own, in any order, on any thread.
 *   - Box-Muller (Box and Muller, 1958) in fp64: element 2j takes r*cos(t), element 2j+1 takes r*sin(t),
 *     with r = sqrt(-2 ln u1), t = 2*pi*u2, u1 = U(draw 2j), u2 = U(draw 2j+1), U(z) = ((z >> 11) + 0.5) / 2^53.
 *   - value = mean + std * z in fp64, rounded to fp32, then to fp16 with round-to-nearest-even.
 *   - Token ids: draw i mod vocab.
 *   - FP8 expert weights (the sparse-MoE model): fp32 values as above, quantised per row to E4M3 with a
 *     fp32 scale (synth_e4m3_rows); the model's weight is the E4M3 value times the row's scale.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_base(uint64_t seed, uint64_t tensor_id) {
  return sm64_mix(sm64_mix(seed + GOLDEN) ^ (tensor_id * 0xD1B54A32D192ED03ULL));
}

static inline uint64_t draw(uint64_t base, uint64_t i) { return sm64_mix(base + (i + 1) * GOLDEN); }

static inline double unit_open(uint64_t z) { return ((double)(z >> 11) + 0.5) * (1.0 / 9007199254740992.0); }

/* fp32 -> binary16 bits, round to nearest, ties to even. */
static uint16_t to_half_bits(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) return (uint16_t)(sign | (ax > 0x7F800000u ? 0x7E00u : 0x7C00u));
  if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* >= 65520 rounds to infinity */
  if (ax < 0x38800000u) {                                     /* below 2^-14: subnormal result */
    if (ax < 0x33000000u) return (uint16_t)sign;               /* below 2^-25: rounds to zero */
    uint32_t e = ax >> 23;
    uint32_t m = (ax & 0x7FFFFFu) | 0x800000u;
    uint32_t shift = 126u - e; /* value / 2^-24 = m * 2^(e-126) */
    uint32_t q = m >> shift, rem = m & ((1u << shift) - 1u), half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (q & 1u))) q++;
    return (uint16_t)(sign | q);
  }
  uint32_t q = (ax >> 13) - (112u << 10);
  uint32_t rem = ax & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q++;
  return (uint16_t)(sign | q);
}

static inline double normal_at(uint64_t base, uint64_t i) {
  uint64_t j = i >> 1;
  double u1 = unit_open(draw(base, 2 * j)), u2 = unit_open(draw(base, 2 * j + 1));
  double r = sqrt(-2.0 * log(u1)), t = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(t) : r * cos(t);
}

/* out[i] = fp16(fp32(mean + std * N_i)) for i in [0, n). */
void synth_normal_f16(uint64_t seed, uint64_t tensor_id, int64_t n, double mean, double std, uint16_t *out) {
  uint64_t base = stream_base(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = to_half_bits((float)(mean + std * normal_at(base, (uint64_t)i)));
}

/* out[i] = fp32(mean + std * N_i): used where an input is fp32 (tests of single steps). */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, int64_t n, double mean, double std, float *out) {
  uint64_t base = stream_base(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(mean + std * normal_at(base, (uint64_t)i));
}

/* out[i] = draw(i) mod modulo: uniform token ids. */
void synth_tokens(uint64_t seed, uint64_t tensor_id, int64_t n, int64_t modulo, int32_t *out) {
  uint64_t base = stream_base(seed, tensor_id);
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(draw(base, (uint64_t)i) % (uint64_t)modulo);
}

/* fp32 -> OCP FP8 E4M3 ("fn" variant: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 * largest finite 448, NaN 0x7F), round to nearest with ties to even, saturating at +-448. */
static uint8_t to_e4m3(float f) {
  if (isnan(f)) return 0x7F;
  const uint8_t sign = signbit(f) ? 0x80 : 0;
  const double a = fabs((double)f);
  if (a >= 448.0) return sign | 0x7E;
  if (a < 0.015625) return sign | (uint8_t)rint(a * 512.0); /* below 2^-6: steps of 2^-9; 8 is code 0x08 */
  int e;
  const double m = frexp(a, &e); /* a = m 2^e, 0.5 <= m < 1 */
  int E = e - 1;                  /* a = (1 + frac) 2^E, E in [-6, 8] */
  double q = rint((2.0 * m - 1.0) * 8.0);
  if (q == 8.0) {
    q = 0.0;
    E += 1;
  }
  if (E > 8 || (E == 8 && q > 6.0)) return sign | 0x7E;
  return sign | (uint8_t)(((E + 7) << 3) | (int)q);
}

/* Rows of an FP8 weight matrix with a per-row fp32 scale: w = fp32(std * N_i) for element i = r * cols + c,
 * scale[r] = max_c |w| / 448 (1 if the row is zero), q[r][c] = E4M3(w / scale[r]). The stored model weight is
 * then E4M3(q) * scale[r]. */
void synth_e4m3_rows(uint64_t seed, uint64_t tensor_id, int64_t rows, int64_t cols, double std, uint8_t *q,
                     float *scale) {
  uint64_t base = stream_base(seed, tensor_id);
#pragma omp parallel
  {
    float *w = (float *)malloc((size_t)cols * sizeof(float));
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      float amax = 0.f;
      for (int64_t c = 0; c < cols; ++c) {
        w[c] = (float)(std * normal_at(base, (uint64_t)(r * cols + c)));
        amax = fmaxf(amax, fabsf(w[c]));
      }
      const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
      scale[r] = sc;
      for (int64_t c = 0; c < cols; ++c) q[r * cols + c] = to_e4m3(w[c] / sc);
    }
    free(w);
  }
}

uint8_t synth_f32_to_e4m3(float f) { return to_e4m3(f); }

/* Raw access for the generator's own tests. */
uint64_t synth_draw(uint64_t seed, uint64_t tensor_id, uint64_t i) { return draw(stream_base(seed, tensor_id), i); }
uint64_t synth_splitmix64_next(uint64_t *state) {
  *state += GOLDEN;
  return sm64_mix(*state);
}
uint16_t synth_f32_to_f16(float f) { return to_half_bits(f); }
