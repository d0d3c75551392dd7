// gather.cu — the parameter AllGather's result assembled on one GPU: slot j of
// the flat parameter buffer receives rank j's updated shard, bit for bit
// ("从 Data Parallel 到 ZeRO/FSDP", "ZeRO Stage 1": all-gather the updated
// parameter shards so that every rank again holds identical full parameters).
// A plain multi-source copy: 2 x slot bytes of HBM traffic per copied slot.
// 32-byte loads and stores where every pointer and the slot size allow (on
// GB300 they measured 0.975 / 0.992 of the copy bandwidth on the Llama-7B /
// Qwen2.5-3B flat buffers against 0.954 / 0.951 with 16-byte accesses, both
// with 8 blocks per SM; the launch shape below), else 16-byte, else bytes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"
#include "overlap.cuh"
#include "zs_internal.h"

namespace zs {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;

struct GatherArgs {
  const unsigned char* src[ZS_MAX_WORLD];
  int32_t slot[ZS_MAX_WORLD];
  unsigned char* dst;
  int64_t slot_bytes;
  int32_t world;       // checked build: dst holds world slots
  unsigned int* err;   // checked build: the device error word
};

// Checked build: a unit of `u` bytes at byte `off` of a slot lies inside the
// slot, and the slot inside the world's buffer.
__device__ __forceinline__ bool unit_ok(const GatherArgs& a, int64_t off, int64_t u) {
  return within(off, off + u, 0, a.slot_bytes, a.err) &&
         within(a.slot[blockIdx.y], a.slot[blockIdx.y] + 1, 0, a.world, a.err);
}

__device__ __forceinline__ uint4 ld_once(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// blockIdx.y = active slot; 16-byte units, kUnroll loads in flight per thread.
__global__ void __launch_bounds__(kThreads) gather16_kernel(const __grid_constant__ GatherArgs a) {
  overlap_wait();
  const uint4* src = reinterpret_cast<const uint4*>(a.src[blockIdx.y]);
  uint4* dst = reinterpret_cast<uint4*>(a.dst + (int64_t)a.slot[blockIdx.y] * a.slot_bytes);
  const int64_t n = a.slot_bytes / 16;
  const int64_t stride = (int64_t)gridDim.x * kThreads * kUnroll;
  for (int64_t base = (int64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; base < n;
       base += stride) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = base + (int64_t)u * kThreads;
      if (i < n && unit_ok(a, 16 * i, 16)) r[u] = ld_once(src + i);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = base + (int64_t)u * kThreads;
      if (i < n && unit_ok(a, 16 * i, 16)) dst[i] = r[u];
    }
  }
}

__device__ __forceinline__ void ld32_once(const void* p, uint32_t* r) {
  asm("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "l"(p));
}
__device__ __forceinline__ void st32(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
// blockIdx.y = active slot; 32-byte units, kUnroll loads in flight per thread.
__global__ void __launch_bounds__(kThreads) gather32_kernel(const __grid_constant__ GatherArgs a) {
  overlap_wait();
  const unsigned char* src = a.src[blockIdx.y];
  unsigned char* dst = a.dst + (int64_t)a.slot[blockIdx.y] * a.slot_bytes;
  const int64_t n = a.slot_bytes / 32;
  const int64_t stride = (int64_t)gridDim.x * kThreads * kUnroll;
  for (int64_t base = (int64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; base < n;
       base += stride) {
    uint32_t r[kUnroll][8];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = base + (int64_t)u * kThreads;
      if (i < n && unit_ok(a, 32 * i, 32)) ld32_once(src + 32 * i, r[u]);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = base + (int64_t)u * kThreads;
      if (i < n && unit_ok(a, 32 * i, 32)) st32(dst + 32 * i, r[u]);
    }
  }
}

// Any alignment: byte copy (slots whose byte size is not a multiple of 16).
__global__ void __launch_bounds__(kThreads) gather1_kernel(const __grid_constant__ GatherArgs a) {
  overlap_wait();
  const unsigned char* src = a.src[blockIdx.y];
  unsigned char* dst = a.dst + (int64_t)a.slot[blockIdx.y] * a.slot_bytes;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < a.slot_bytes; i += stride)
    if (unit_ok(a, i, 1)) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_gather(const GatherLaunch& in, cudaStream_t stream) {
  GatherArgs a;
  int active = 0;
  for (int j = 0; j < in.world; ++j) {
    if (!in.srcs[j]) continue;
    a.src[active] = in.srcs[j];
    a.slot[active] = j;
    ++active;
  }
  if (active == 0) return cudaSuccess;
  a.dst = in.dst;
  a.slot_bytes = in.slot_bytes;
  a.world = in.world;
  a.err = ZS_BOUNDS_CHECK ? device_error_word() : nullptr;
  if (ZS_BOUNDS_CHECK && !a.err) return cudaErrorInvalidSymbol;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const bool vec = in.slot_bytes % 16 == 0;
  const int64_t units = vec ? in.slot_bytes / 16 / kUnroll : in.slot_bytes;
  int64_t want = (units + kThreads - 1) / kThreads;
  // Two blocks per SM spread over the active slots, two loads in flight per
  // thread: on GB300 (CUDA graphs of back-to-back gathers) 0.973 / 1.015 /
  // 1.015 of the copy bandwidth for GPT-2-small / Qwen2.5-3B / Llama-7B,
  // against 0.962 / 0.991 / 0.987 with eight blocks and four loads, and 0.87 /
  // 0.92 / 0.92 with four blocks and two loads (plain copies of these sizes
  // show the same shape dependence).
  int64_t cap = ((int64_t)sms * 2 + active - 1) / active;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  dim3 grid((unsigned)want, (unsigned)active);
  bool v32 = in.slot_bytes % 32 == 0 && (uintptr_t)in.dst % 32 == 0;
  for (int k = 0; k < active && v32; ++k) v32 = (uintptr_t)a.src[k] % 32 == 0;
  if (v32) {
    int64_t w32 = (in.slot_bytes / 32 / kUnroll + kThreads - 1) / kThreads;
    if (w32 > cap) w32 = cap;
    if (w32 < 1) w32 = 1;
    return launch_kernel(gather32_kernel, dim3((unsigned)w32, (unsigned)active), dim3(kThreads), 0,
                         stream, a);
  }
  if (vec) return launch_kernel(gather16_kernel, grid, dim3(kThreads), 0, stream, a);
  return launch_kernel(gather1_kernel, grid, dim3(kThreads), 0, stream, a);
}

}  // namespace zs
