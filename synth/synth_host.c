/*
 * synth_host.c — host side of the synthetic input generator (see synth.h for
 * the definition). Fills are split over POSIX threads; every element depends
 * only on its own counter key, so the result does not depend on the split.
 * Compiled with -O2 -ffp-contract=off.
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

static void* syn_worker(void* arg) {
  syn_job* j = (syn_job*)arg;
  for (int64_t i = j->begin; i < j->end; ++i) {
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
