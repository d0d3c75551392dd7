// accum.cu — gradient accumulation on the shard.
//
// "从 Data Parallel 到 ZeRO/FSDP", "Gradient Accumulation 会改变生命周期": with
// G > 1 micro-batches per optimizer step, a sharded job must settle whether
// every micro-step ReduceScatters, whether gradients accumulate on the shard
// or on the full tensor, and whether the loss is divided by G; "ZeRO vs FSDP:
// A Rigorous Dissection", §7 (gradient accumulation): communication belongs to
// the last micro-batch only when the full tensor is accumulated. Here the
// ZeRO-2/3 choice: every micro-step's ReduceScatter output (the N slices of
// this rank's shard) is reduced to its mean and added into an fp32 shard
// accumulator (zs_grad_accumulate: 2N + 8 bytes per element, 2N + 4 on the
// first micro-step, which overwrites); the last micro-step's slices go straight
// into the step, which forms ((accumulator + mean) * (1/G)): the average over
// the G micro-batches (the loss divided by G) — zs_shard_step_accumulated,
// 2N + 30 bytes per element, the shared kernel template with ACC = true.
#include <cuda_runtime.h>
#include <stdint.h>

#include "step_kernel.cuh"
#include "zs_internal.h"

namespace zs {
namespace {

// accum[i] = (first ? 0 : accum[i]) + mean_j(x_j[i]), the mean formed exactly
// as the step forms it. GW = 16/8: vector groups; 0: element by element.
template <int GW, bool BF16G, int MAXN>
__global__ void __launch_bounds__(kThreads, 2)
    accumulate_kernel(const __grid_constant__ StepArgs<MAXN> a, int first) {
  overlap_wait();
  float* accum = const_cast<float*>(a.accum);  // the output of this kernel
  const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  auto one = [&](int64_t i) {
    if (!within(i, i + 1, a.win_lo, a.win_hi, a.err)) return;
    float acc = 0.0f;
    for (int j = 0; j < a.world; ++j) {
      const float x = BF16G ? __uint_as_float(
                                  (uint32_t) static_cast<const uint16_t*>(a.grads[j])[i] << 16)
                            : static_cast<const float*>(a.grads[j])[i];
      acc = __fadd_rn(acc, x);
    }
    accum[i] = __fadd_rn(first ? 0.0f : accum[i], __fmul_rn(acc, a.s.invN));
  };
  int64_t g0 = 0, g1 = 0;
  if constexpr (GW > 0) {
    g0 = (a.lo + GW - 1) / GW;
    g1 = a.hi / GW;
  }
  if (g0 >= g1) {
    for (int64_t i = a.lo + tid; i < a.hi; i += stride) one(i);
    return;
  }
  if constexpr (GW > 0) {
    const int64_t head = g0 * GW - a.lo, tail = a.hi - g1 * GW;
    if (tid < head) one(a.lo + tid);
    else if (tid < head + tail) one(g1 * GW + (tid - head));
    for (int64_t g = g0 + tid; g < g1; g += stride) {
      if (!within(GW * g, GW * g + GW, a.win_lo, a.win_hi, a.err)) continue;
      float prev[GW], acc[GW];
      if (!first) load_state<GW>(accum + GW * g, prev);
      reduce_group<GW, BF16G>(a, g, acc);
#pragma unroll
      for (int k = 0; k < GW; ++k)
        acc[k] = __fadd_rn(first ? 0.0f : prev[k], __fmul_rn(acc[k], a.s.invN));
      store_state<GW>(accum + GW * g, acc);
    }
  }
}

template <int GW, bool BF16G, int MAXN>
cudaError_t launch_acc(const ShardStepLaunch& in, int first, cudaStream_t stream) {
  static std::atomic<int> max_blocks_by_dev[64];
  auto kernel = accumulate_kernel<GW, BF16G, MAXN>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int max_blocks = max_blocks_by_dev[dev & 63].load(std::memory_order_relaxed);
  if (max_blocks == 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
    if (e != cudaSuccess) return e;
    max_blocks = 2 * sms * (per_sm > 0 ? per_sm : 1);
    max_blocks_by_dev[dev & 63].store(max_blocks, std::memory_order_relaxed);
  }
  StepArgs<MAXN> a;
  for (int j = 0; j < MAXN; ++j) a.grads[j] = j < in.world ? in.grads[j] : nullptr;
  a.master = nullptr;
  a.m = nullptr;
  a.v = nullptr;
  a.slot = nullptr;
  a.lo = in.lo;
  a.hi = in.hi;
  a.world = in.world;
  a.coef = nullptr;
  a.skip = nullptr;
  a.accum = in.accum;
  a.invG = 1.0f;
  a.s = in.s;
  a.win_lo = in.win.lo;
  a.win_hi = in.win.hi;
  a.err = ZS_BOUNDS_CHECK ? device_error_word() : nullptr;
  if (ZS_BOUNDS_CHECK && !a.err) return cudaErrorInvalidSymbol;
  const int64_t units = GW > 0 ? (in.hi - in.lo) / GW + 2 : (in.hi - in.lo);
  int64_t blocks = (units + kThreads - 1) / kThreads;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  return launch_kernel(kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, a, first);
}

template <bool BF16G>
cudaError_t dispatch_acc(const ShardStepLaunch& a, int first, cudaStream_t stream) {
  if (a.vec_width == 16) {
    if (a.world <= 16) return launch_acc<16, BF16G, 16>(a, first, stream);
    return launch_acc<16, BF16G, ZS_MAX_WORLD>(a, first, stream);
  }
  if (a.vec_width == 8) return launch_acc<8, BF16G, ZS_MAX_WORLD>(a, first, stream);
  return launch_acc<0, BF16G, ZS_MAX_WORLD>(a, first, stream);
}

}  // namespace

cudaError_t launch_grad_accumulate(const ShardStepLaunch& a, int first, cudaStream_t stream) {
  return a.grad_dtype == ZS_BF16 ? dispatch_acc<true>(a, first, stream)
                                 : dispatch_acc<false>(a, first, stream);
}

cudaError_t launch_shard_step_accumulated(const ShardStepLaunch& a, cudaStream_t stream) {
  return launch_step_kernel<true>(a, stream);
}

}  // namespace zs
