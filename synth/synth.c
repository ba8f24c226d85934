/*
 * Seeded synthetic input generator shared by the tests, the oracle checks and
 * the benchmark.  It produces the raw *fields* of a workload -- integer codes,
 * 4-bit sub-block scales/mins, fp16 scale bit patterns, bf16 activations and
 * fp32 router weights -- and nothing else.  It knows no block layout, no
 * dequantisation rule and no part of the MoE arithmetic: turning fields into
 * Q4_1 / Q2_K block bytes is done separately by each consumer.
 *
 * Randomness is counter based: value i of a stream is SplitMix64 evaluated at
 * state key + (i + 1) * 0x9E3779B97F4A7C15, i.e. the (i+1)-th output of the
 * SplitMix64 generator started from `key` (G. Steele, D. Lea, C. Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014; finaliser
 * constants as published with S. Vigna's splitmix64.c).  Any element can be
 * regenerated on demand, in any order, on any thread.
 *
 * Normals use the Box-Muller transform in double precision (one normal per
 * pair of uniforms, cosine branch), then round-to-nearest-even into the
 * requested storage format.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Value i of the stream keyed by `key`. */
uint64_t synth_u64(uint64_t key, uint64_t i) {
  return sm64_mix(key + (i + 1) * GOLDEN_GAMMA);
}

/* Stream key for (seed, layer, tensor, expert, field). */
uint64_t synth_key(uint64_t seed, uint64_t layer, uint64_t tensor,
                   uint64_t expert, uint64_t field) {
  uint64_t k = sm64_mix(seed + GOLDEN_GAMMA);
  k = sm64_mix(k ^ (layer * 0xD1B54A32D192ED03ULL));
  k = sm64_mix(k ^ (tensor * 0xAEF17502108EF2D9ULL));
  k = sm64_mix(k ^ (expert * 0xDB4F0B9175AE2165ULL));
  k = sm64_mix(k ^ (field * 0xCB24D0A5C88C35B3ULL));
  return k;
}

/* Uniform double in (0, 1]: 53 random bits. */
static inline double u01(uint64_t v) {
  return (double)((v >> 11) + 1) * (1.0 / 9007199254740992.0);
}

/* Standard normal number i of the stream (uses u64 values 2i and 2i+1). */
double synth_normal(uint64_t key, uint64_t i) {
  double u1 = u01(synth_u64(key, 2 * i));
  double u2 = u01(synth_u64(key, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* Integer codes uniform in [0, 2^bits), bits in 1..8: element i takes bits
 * [bits*(i % per), ...) of u64 number i / per, per = 64 / bits. */
void synth_codes(uint64_t key, int64_t start, int64_t n, int bits,
                 uint8_t *out) {
  const int per = 64 / bits;
  const uint64_t mask = (1ULL << bits) - 1ULL;
  if (n <= 0) return;
  const int64_t w0 = start / per, w1 = (start + n - 1) / per; /* u64 words touched */
#pragma omp parallel for schedule(static)
  for (int64_t w = w0; w <= w1; ++w) {
    uint64_t v = synth_u64(key, (uint64_t)w);
    int64_t i0 = w * per, i1 = i0 + per;
    if (i0 < start) i0 = start;
    if (i1 > start + n) i1 = start + n;
    for (int64_t i = i0; i < i1; ++i)
      out[i - start] = (uint8_t)((v >> (bits * (int)(i - w * per))) & mask);
  }
}

/* Round a double to a binary format with `p` significand bits (incl. the
 * implicit one), minimum normal exponent `emin` and maximum exponent `emax`,
 * round-to-nearest-even, returning the rounded value as a double. */
static double round_to_format(double v, int p, int emin, int emax) {
  if (v == 0.0 || isnan(v) || isinf(v)) return v;
  int e;
  double m = frexp(fabs(v), &e);          /* |v| = m * 2^e, m in [0.5, 1) */
  int exp_unbiased = e - 1;                /* |v| = 1.m * 2^exp_unbiased */
  int q = exp_unbiased < emin ? emin : exp_unbiased; /* quantum exponent */
  double scaled = ldexp(fabs(v), (p - 1) - q);       /* exact (power of 2) */
  double r = nearbyint(scaled);            /* default mode: ties to even */
  double out = ldexp(r, q - (p - 1));
  if (out >= ldexp(2.0, emax)) out = INFINITY;
  (void)m;
  return v < 0 ? -out : out;
}

/* Bit pattern of an already-representable fp16 value. */
static uint16_t f16_bits_of(double v) {
  uint16_t s = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (isnan(v)) return 0x7E00;
  if (isinf(a)) return s | 0x7C00;
  if (a == 0.0) return s;
  int e;
  frexp(a, &e);
  int ex = e - 1;
  if (ex < -14) { /* subnormal: a = frac * 2^-24 */
    return s | (uint16_t)ldexp(a, 24);
  }
  uint16_t frac = (uint16_t)(ldexp(a, 10 - ex) - 1024.0);
  return s | (uint16_t)((ex + 15) << 10) | frac;
}

/* Bit pattern of an already-representable bf16 value (via fp32 bits). */
static uint16_t bf16_bits_of(double v) {
  float f = (float)v; /* exact: v has at most 8 significand bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

uint16_t synth_round_f16(double v) { return f16_bits_of(round_to_format(v, 11, -14, 15)); }
uint16_t synth_round_bf16(double v) { return bf16_bits_of(round_to_format(v, 8, -126, 127)); }
float synth_round_f32(double v) { return (float)round_to_format(v, 24, -126, 127); }

/* |N(0, sigma)| rounded to fp16; out[j] for stream elements start..start+n. */
void synth_abs_normal_f16(uint64_t key, int64_t start, int64_t n, double sigma,
                          uint16_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j)
    out[j] = synth_round_f16(fabs(sigma * synth_normal(key, (uint64_t)(start + j))));
}

/* scale * N(0, sigma) rounded to bf16. */
void synth_normal_bf16(uint64_t key, int64_t start, int64_t n, double sigma,
                       uint16_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j)
    out[j] = synth_round_bf16(sigma * synth_normal(key, (uint64_t)(start + j)));
}

/* N(0, sigma) rounded to fp32. */
void synth_normal_f32(uint64_t key, int64_t start, int64_t n, double sigma,
                      float *out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j)
    out[j] = synth_round_f32(sigma * synth_normal(key, (uint64_t)(start + j)));
}

/* out[j] = fp16(mult * value of fp16 pattern in[j]) for a power-of-two
 * multiplier (used for "min = -8 d" style derived fields; exact unless the
 * result overflows fp16). */
void synth_f16_scale_pow2(const uint16_t *in, int64_t n, double mult,
                          uint16_t *out) {
  for (int64_t j = 0; j < n; ++j) {
    uint16_t h = in[j];
    int ex = (h >> 10) & 31, fr = h & 1023;
    double v = ex == 0 ? ldexp((double)fr, -24)
                       : ldexp((double)(fr | 1024), ex - 25);
    if (ex == 31) v = fr ? NAN : INFINITY;
    if (h & 0x8000) v = -v;
    out[j] = synth_round_f16(mult * v);
  }
}
