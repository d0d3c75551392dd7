/*
 * synth.h — seeded, counter-based synthetic inputs for the shard-local step.
 *
 * This module only makes inputs (fp32 master weights, bf16/fp32 incoming
 * gradient slices). It holds none of the step's arithmetic: no reduction,
 * no optimizer update, no layout. Both the CPU oracle's tests and the CUDA
 * path's tests/bench draw their inputs from here, so that both sides see the
 * same bits.
 *
 * Definition (the same on host and device; every operation is an integer op
 * or an IEEE-754 double +, -, *, / or sqrt, so gcc with -ffp-contract=off and
 * nvcc with -fmad=false produce bit-identical values):
 *
 *   mix64(z)      SplitMix64 finaliser (Steele, Lea & Flood, "Fast splittable
 *                 pseudorandom number generators", OOPSLA 2014).
 *   key(seed, stream, step, rank, index)
 *                 h = mix64(seed + G*(stream+1)); then for f in (step, rank,
 *                 index): h = mix64(h + G + f).   G = 0x9E3779B97F4A7C15.
 *   unit(r)       (r >> 11) * 2^-52 - 1, uniform on [-1, 1).
 *   normal(key)   Marsaglia polar method: for attempt a = 0..63,
 *                 u = unit(mix64(key + (2a+1)G)), v = unit(mix64(key + (2a+2)G)),
 *                 s = u*u + v*v; accept when 0 < s < 1 and return
 *                 u * sqrt((-2 * ln(s)) / s). After 64 rejections return 0.
 *   ln(x)         x = m * 2^e with m in [1/sqrt2, sqrt2); t = (m-1)/(m+1);
 *                 ln(m) = 2t * sum_{k=0}^{12} t^{2k}/(2k+1)   (the atanh series,
 *                 Abramowitz & Stegun 4.1.27), evaluated by Horner from k=12;
 *                 ln(x) = 2t*S + e*ln2.
 *   value         x = sigma * normal(key(seed, stream, step, rank, index));
 *                 if an outlier fraction f > 0 is given and
 *                 mix-key(seed, OUTLIER, step, rank, index) < f * 2^64 then
 *                 x = x * outlier_scale; the sample is (float)x (round to
 *                 nearest even), and a bf16 sample is that float rounded to
 *                 bf16 (nearest even, by this module's own conversion).
 *                 Indices >= p_limit (the flat buffer's tail pad) give +0.
 *
 * `index` is the element's GLOBAL flat index, so a tensor's values do not
 * depend on how it is sharded; `rank` is the source rank whose local gradient
 * is drawn; `step` is the optimizer step t.
 */
#ifndef ZS_SYNTH_H
#define ZS_SYNTH_H

#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef __CUDACC__
#define SYN_FN __host__ __device__ static inline
#else
#define SYN_FN static inline
#endif

#define SYN_STREAM_MASTER 1u
#define SYN_STREAM_GRAD 2u
#define SYN_STREAM_OUTLIER 3u

#define SYN_GOLDEN 0x9E3779B97F4A7C15ull
#define SYN_MAX_ATTEMPTS 64u

SYN_FN uint64_t syn_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

SYN_FN uint64_t syn_key(uint64_t seed, uint64_t stream, uint64_t step,
                        uint64_t rank, uint64_t index) {
  uint64_t h = syn_mix64(seed + SYN_GOLDEN * (stream + 1u));
  h = syn_mix64(h + SYN_GOLDEN + step);
  h = syn_mix64(h + SYN_GOLDEN + rank);
  h = syn_mix64(h + SYN_GOLDEN + index);
  return h;
}

SYN_FN double syn_unit(uint64_t r) {
  return (double)(r >> 11) * (1.0 / 4503599627370496.0) - 1.0; /* 2^-52 */
}

/* Natural log of a positive normal double (the generator's own, see above). */
SYN_FN double syn_log(double x) {
  uint64_t b;
  memcpy(&b, &x, sizeof b);
  int64_t e = (int64_t)((b >> 52) & 0x7FFu) - 1023;
  b = (b & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull;
  double m;
  memcpy(&m, &b, sizeof m);
  if (m > 1.4142135623730951) {
    m = m * 0.5;
    e = e + 1;
  }
  double t = (m - 1.0) / (m + 1.0);
  double t2 = t * t;
  double s = 1.0 / 25.0;
  for (int k = 11; k >= 0; --k) s = s * t2 + 1.0 / (double)(2 * k + 1);
  return (2.0 * t) * s + (double)e * 0.69314718055994530942;
}

SYN_FN double syn_normal(uint64_t key) {
  for (uint64_t a = 0; a < SYN_MAX_ATTEMPTS; ++a) {
    double u = syn_unit(syn_mix64(key + (2u * a + 1u) * SYN_GOLDEN));
    double v = syn_unit(syn_mix64(key + (2u * a + 2u) * SYN_GOLDEN));
    double s = u * u + v * v;
    if (s > 0.0 && s < 1.0) return u * sqrt((-2.0 * syn_log(s)) / s); /* IEEE, correctly rounded */
  }
  return 0.0;
}

typedef struct {
  uint64_t seed;
  uint32_t stream;
  uint64_t step;
  uint64_t rank;
  int64_t p_limit;        /* indices >= p_limit give 0 */
  double sigma;
  uint64_t outlier_thr;   /* 0 = no outliers */
  double outlier_scale;
} syn_params;

SYN_FN float syn_value(const syn_params* q, int64_t index) {
  if (index >= q->p_limit || index < 0) return 0.0f;
  double x = q->sigma *
             syn_normal(syn_key(q->seed, q->stream, q->step, q->rank, (uint64_t)index));
  if (q->outlier_thr != 0u &&
      syn_key(q->seed, SYN_STREAM_OUTLIER, q->step, q->rank, (uint64_t)index) <
          q->outlier_thr)
    x = x * q->outlier_scale;
  return (float)x;
}

/* Round a float to bf16, nearest even; NaN becomes a quiet NaN. */
SYN_FN uint16_t syn_to_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, sizeof b);
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu) != 0u)
    return (uint16_t)((b >> 16) | 0x0040u);
  uint32_t keep = b >> 16;
  uint32_t rest = b & 0xFFFFu;
  if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
  return (uint16_t)keep;
}

#endif /* ZS_SYNTH_H */
