/*
 * synth_dev.cu — device side of the synthetic input generator (see synth.h).
 * Fills a device buffer with exactly the values the host side produces for
 * the same arguments (compiled with -fmad=false; double ops are IEEE).
 * Used to put full-size benchmark inputs into HBM without a host round trip.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth.h"

extern "C" uint64_t syn_threshold_host(double frac);

template <bool BF16>
__global__ void syn_fill_kernel(void* __restrict__ out, int64_t n, int64_t index0,
                                syn_params q) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float x = syn_value(&q, index0 + i);
    if (BF16)
      static_cast<uint16_t*>(out)[i] = syn_to_bf16(x);
    else
      static_cast<float*>(out)[i] = x;
  }
}

static int syn_launch(void* out, int bf16, int64_t n, int64_t index0, uint64_t seed,
                      uint32_t stream_id, uint64_t step, uint64_t rank, double sigma,
                      int64_t p_limit, double outlier_frac, double outlier_scale,
                      void* cuda_stream) {
  if (n < 0 || (n > 0 && !out)) return -1;
  if (n == 0) return 0;
  syn_params q;
  q.seed = seed;
  q.stream = stream_id;
  q.step = step;
  q.rank = rank;
  q.p_limit = p_limit;
  q.sigma = sigma;
  q.outlier_thr = syn_threshold_host(outlier_frac);
  q.outlier_scale = outlier_scale;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -2;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -2;
  const int threads = 256;
  int64_t want = (n + threads - 1) / threads;
  int64_t cap = (int64_t)sms * 8;
  int blocks = (int)(want < cap ? want : cap);
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  if (bf16)
    syn_fill_kernel<true><<<blocks, threads, 0, s>>>(out, n, index0, q);
  else
    syn_fill_kernel<false><<<blocks, threads, 0, s>>>(out, n, index0, q);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

extern "C" int syn_fill_f32_dev(float* out, int64_t n, int64_t index0, uint64_t seed,
                                uint32_t stream_id, uint64_t step, uint64_t rank,
                                double sigma, int64_t p_limit, double outlier_frac,
                                double outlier_scale, void* cuda_stream) {
  return syn_launch(out, 0, n, index0, seed, stream_id, step, rank, sigma, p_limit,
                    outlier_frac, outlier_scale, cuda_stream);
}

extern "C" int syn_fill_bf16_dev(uint16_t* out, int64_t n, int64_t index0, uint64_t seed,
                                 uint32_t stream_id, uint64_t step, uint64_t rank,
                                 double sigma, int64_t p_limit, double outlier_frac,
                                 double outlier_scale, void* cuda_stream) {
  return syn_launch(out, 1, n, index0, seed, stream_id, step, rank, sigma, p_limit,
                    outlier_frac, outlier_scale, cuda_stream);
}
