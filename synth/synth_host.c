/*
 * synth_host.c — host side of the synthetic input generator (see synth.h for
 * the definition). Fills are split over POSIX threads; every element depends
 * only on its own counter key, so the result does not depend on the split.
 * Compiled with -O2 -ffp-contract=off.
 *
 * Contiguous fills run SYN_LANES elements in lockstep: the first attempt of
 * the polar method, its logarithm and square root for all lanes at once
 * (independent chains the compiler can interleave and vectorise, and no
 * data-dependent branch), then the rare lanes whose first pair was rejected
 * continue one by one with attempt 1 of the scalar definition. Every lane
 * performs exactly the IEEE operations of synth.h in the same order, so the
 * values are the definition's bits; gathers at arbitrary indices use the
 * scalar definition directly, and the tests compare the two.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#include "synth.h"

typedef struct {
  syn_params q;
  int64_t index0;
  const int64_t* idx; /* NULL: contiguous from index0 */
  void* out;
  int bf16;
  int64_t begin, end;
} syn_job;

#define SYN_LANES 16

/* The key prefix shared by every index of one (seed, stream, step, rank):
 * syn_key(seed, stream, step, rank, index) = mix64(prefix + G + index). */
static uint64_t syn_prefix(uint64_t seed, uint64_t stream, uint64_t step, uint64_t rank) {
  uint64_t h = syn_mix64(seed + SYN_GOLDEN * (stream + 1u));
  h = syn_mix64(h + SYN_GOLDEN + step);
  return syn_mix64(h + SYN_GOLDEN + rank);
}

/* The polar method from attempt a0 on (synth.h's syn_normal, resumed). */
static double syn_normal_from(uint64_t key, uint64_t a0) {
  for (uint64_t a = a0; a < SYN_MAX_ATTEMPTS; ++a) {
    double u = syn_unit(syn_mix64(key + (2u * a + 1u) * SYN_GOLDEN));
    double v = syn_unit(syn_mix64(key + (2u * a + 2u) * SYN_GOLDEN));
    double s = u * u + v * v;
    if (s > 0.0 && s < 1.0) return u * sqrt((-2.0 * syn_log(s)) / s);
  }
  return 0.0;
}

/* SYN_LANES values at global indices first .. first + SYN_LANES - 1. */
static void syn_lanes(const syn_params* q, uint64_t pre, uint64_t pre_out, int64_t first,
                      void* out, int bf16) {
  double u[SYN_LANES], s[SYN_LANES], m[SYN_LANES], e[SYN_LANES], t[SYN_LANES],
      t2[SYN_LANES], h[SYN_LANES], x[SYN_LANES];
  uint64_t key[SYN_LANES];
  int ok[SYN_LANES];
  for (int k = 0; k < SYN_LANES; ++k) {
    key[k] = syn_mix64(pre + SYN_GOLDEN + (uint64_t)(first + k));
    u[k] = syn_unit(syn_mix64(key[k] + SYN_GOLDEN));
    double v = syn_unit(syn_mix64(key[k] + 2u * SYN_GOLDEN));
    s[k] = u[k] * u[k] + v * v;
    ok[k] = s[k] > 0.0 && s[k] < 1.0;
    if (!ok[k]) s[k] = 0.5; /* any value in range; the lane is redone below */
  }
  /* syn_log on every lane: the same operations, the branch as a select. */
  for (int k = 0; k < SYN_LANES; ++k) {
    uint64_t b;
    memcpy(&b, &s[k], sizeof b);
    int64_t ex = (int64_t)((b >> 52) & 0x7FFu) - 1023;
    b = (b & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull;
    double mm;
    memcpy(&mm, &b, sizeof mm);
    int big = mm > 1.4142135623730951;
    m[k] = big ? mm * 0.5 : mm;
    e[k] = (double)(big ? ex + 1 : ex);
  }
  for (int k = 0; k < SYN_LANES; ++k) {
    t[k] = (m[k] - 1.0) / (m[k] + 1.0);
    t2[k] = t[k] * t[k];
    h[k] = 1.0 / 25.0;
  }
  for (int c = 11; c >= 0; --c) {
    const double inv = 1.0 / (double)(2 * c + 1);
    for (int k = 0; k < SYN_LANES; ++k) h[k] = h[k] * t2[k] + inv;
  }
  for (int k = 0; k < SYN_LANES; ++k) {
    double lg = (2.0 * t[k]) * h[k] + e[k] * 0.69314718055994530942;
    x[k] = u[k] * sqrt((-2.0 * lg) / s[k]);
  }
  for (int k = 0; k < SYN_LANES; ++k) {
    const int64_t index = first + k;
    float val = 0.0f;
    if (index < q->p_limit && index >= 0) {
      double r = q->sigma * (ok[k] ? x[k] : syn_normal_from(key[k], 1u));
      if (q->outlier_thr != 0u &&
          syn_mix64(pre_out + SYN_GOLDEN + (uint64_t)index) < q->outlier_thr)
        r = r * q->outlier_scale;
      val = (float)r;
    }
    if (bf16)
      ((uint16_t*)out)[k] = syn_to_bf16(val);
    else
      ((float*)out)[k] = val;
  }
}

static void* syn_worker(void* arg) {
  syn_job* j = (syn_job*)arg;
  int64_t i = j->begin;
  if (!j->idx) {
    const uint64_t pre = syn_prefix(j->q.seed, j->q.stream, j->q.step, j->q.rank);
    const uint64_t pre_out = syn_prefix(j->q.seed, SYN_STREAM_OUTLIER, j->q.step, j->q.rank);
    const size_t eb = j->bf16 ? 2 : 4;
    for (; i + SYN_LANES <= j->end; i += SYN_LANES)
      syn_lanes(&j->q, pre, pre_out, j->index0 + i, (unsigned char*)j->out + eb * (size_t)i,
                j->bf16);
  }
  for (; i < j->end; ++i) {
    int64_t index = j->idx ? j->idx[i] : j->index0 + i;
    float x = syn_value(&j->q, index);
    if (j->bf16)
      ((uint16_t*)j->out)[i] = syn_to_bf16(x);
    else
      ((float*)j->out)[i] = x;
  }
  return NULL;
}

static uint64_t syn_threshold(double frac) {
  if (!(frac > 0.0)) return 0u;
  if (frac >= 1.0) return UINT64_MAX;
  return (uint64_t)(frac * 18446744073709551616.0); /* frac * 2^64 */
}

static int syn_run(void* out, int bf16, int64_t n, const int64_t* idx, int64_t index0,
                   uint64_t seed, uint32_t stream, uint64_t step, uint64_t rank,
                   double sigma, int64_t p_limit, double outlier_frac,
                   double outlier_scale, int threads) {
  if (n < 0 || (n > 0 && !out)) return -1;
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if ((int64_t)threads > n / 4096 + 1) threads = (int)(n / 4096 + 1);
  syn_params q;
  q.seed = seed;
  q.stream = stream;
  q.step = step;
  q.rank = rank;
  q.p_limit = p_limit;
  q.sigma = sigma;
  q.outlier_thr = syn_threshold(outlier_frac);
  q.outlier_scale = outlier_scale;
  syn_job jobs[256];
  pthread_t tids[256];
  int64_t chunk = (n + threads - 1) / threads;
  for (int t = 0; t < threads; ++t) {
    jobs[t].q = q;
    jobs[t].index0 = index0;
    jobs[t].idx = idx;
    jobs[t].out = out;
    jobs[t].bf16 = bf16;
    jobs[t].begin = (int64_t)t * chunk < n ? (int64_t)t * chunk : n;
    jobs[t].end = (int64_t)(t + 1) * chunk < n ? (int64_t)(t + 1) * chunk : n;
  }
  if (threads == 1) {
    syn_worker(&jobs[0]);
    return 0;
  }
  int started = 0;
  for (int t = 0; t < threads; ++t) {
    if (pthread_create(&tids[t], NULL, syn_worker, &jobs[t]) != 0) break;
    ++started;
  }
  for (int t = started; t < threads; ++t) syn_worker(&jobs[t]);
  for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
  return 0;
}

/* Contiguous fill: out[i] = value(index0 + i). Returns 0, or -1 on bad args. */
int syn_fill_f32(float* out, int64_t n, int64_t index0, uint64_t seed, uint32_t stream,
                 uint64_t step, uint64_t rank, double sigma, int64_t p_limit,
                 double outlier_frac, double outlier_scale, int threads) {
  return syn_run(out, 0, n, NULL, index0, seed, stream, step, rank, sigma, p_limit,
                 outlier_frac, outlier_scale, threads);
}

int syn_fill_bf16(uint16_t* out, int64_t n, int64_t index0, uint64_t seed,
                  uint32_t stream, uint64_t step, uint64_t rank, double sigma,
                  int64_t p_limit, double outlier_frac, double outlier_scale,
                  int threads) {
  return syn_run(out, 1, n, NULL, index0, seed, stream, step, rank, sigma, p_limit,
                 outlier_frac, outlier_scale, threads);
}

/* Gather at arbitrary global indices: out[i] = value(idx[i]). */
int syn_at_f32(float* out, const int64_t* idx, int64_t n, uint64_t seed, uint32_t stream,
               uint64_t step, uint64_t rank, double sigma, int64_t p_limit,
               double outlier_frac, double outlier_scale, int threads) {
  if (n > 0 && !idx) return -1;
  return syn_run(out, 0, n, idx, 0, seed, stream, step, rank, sigma, p_limit,
                 outlier_frac, outlier_scale, threads);
}

int syn_at_bf16(uint16_t* out, const int64_t* idx, int64_t n, uint64_t seed,
                uint32_t stream, uint64_t step, uint64_t rank, double sigma,
                int64_t p_limit, double outlier_frac, double outlier_scale, int threads) {
  if (n > 0 && !idx) return -1;
  return syn_run(out, 1, n, idx, 0, seed, stream, step, rank, sigma, p_limit,
                 outlier_frac, outlier_scale, threads);
}

/* Exposed for tests of the generator itself. */
double syn_log_host(double x) { return syn_log(x); }
uint64_t syn_key_host(uint64_t seed, uint64_t stream, uint64_t step, uint64_t rank,
                      uint64_t index) {
  return syn_key(seed, stream, step, rank, index);
}
uint64_t syn_threshold_host(double frac) { return syn_threshold(frac); }
