// shard_step.cu — the fused shard-local step: N-slice fp32 mean + AdamW on the
// fp32 master/m/v shard + cast of the updated master into this rank's slot of
// the AllGather buffer, in one memory-bound pass.
//
// The step ("从 Data Parallel 到 ZeRO/FSDP", "ZeRO Stage 1": after the gradient
// ReduceScatter the owner rank updates its optimizer/parameter shard, then
// all-gathers the updated parameters; "ZeRO vs FSDP: A Rigorous Dissection",
// §2.1-2.3) touches each shard element once: it reads N incoming gradient
// values and the fp32 master, m and v, and writes master, m, v and one
// low-precision parameter: g*N + 24 + p bytes per element and about N + 15
// flops, so HBM bandwidth bounds it and no tensor-core work exists here.
//
// Layout of the work: the shard-local range [lo, hi) is cut into groups of GW
// elements. A persistent grid walks the groups with a grid stride; a group is
// one thread's vector loads of every slice and of the three states, the fp32
// arithmetic, and vector stores. GW = 16 uses 32-byte accesses (one ld/st.v8
// per 16 bf16 or 8 fp32 values, Blackwell's widest global access): the most
// bytes per load instruction, and enough bytes in flight per SM at two
// resident blocks. GW = 8 uses 16-byte accesses for callers whose pointers
// are only 16-byte aligned. Elements before the first and after the last
// whole group (bucket ranges start and end at tensor boundaries) are done one
// by one, as is everything when the rank's slot is not vector-aligned.
//
// Arithmetic: every operation is an IEEE binary32 op rounded to nearest even
// (the _rn intrinsics are never contracted into FMAs), in the order the
// method fixes, so results are reproducible bit for bit.
//
// The kernel templates live in step_kernel.cuh (shared with the last
// micro-step of gradient accumulation); this file instantiates the step.
#include <cuda_runtime.h>
#include <stdint.h>

#include "step_kernel.cuh"
#include "zs_internal.h"

namespace zs {

// Bit value 1: a check of the bounds-checked build failed; 2: a bounded wait
// gave up. Read and cleared by zs_check_device_error.
__device__ unsigned int g_error_word;

int bounds_checked() { return ZS_BOUNDS_CHECK; }

cudaError_t launch_shard_step(const ShardStepLaunch& a, cudaStream_t stream) {
  return launch_step_kernel<false>(a, stream);
}

namespace {
// A wait that is never satisfied: one mbarrier, initialised and never arrived
// on, waited for through the step kernels' bounded wait with `polls` polls.
__global__ void wait_timeout_kernel(unsigned int* err, uint32_t polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  mbar_wait(&bar, 0, err, polls);
}
}  // namespace

cudaError_t launch_wait_timeout(uint32_t polls, cudaStream_t stream) {
  unsigned int* err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err, polls);
  return cudaGetLastError();
}

unsigned int* device_error_word() {
  static std::atomic<unsigned int*> by_dev[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  unsigned int* w = by_dev[dev & 63].load(std::memory_order_acquire);
  if (!w) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_error_word) != cudaSuccess) return nullptr;
    w = static_cast<unsigned int*>(addr);
    by_dev[dev & 63].store(w, std::memory_order_release);
  }
  return w;
}

cudaError_t read_and_clear_device_error(cudaStream_t stream, unsigned int* word) {
  void* addr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&addr, g_error_word);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpy(word, addr, sizeof(unsigned int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(addr, 0, sizeof(unsigned int));
  return e;
}

}  // namespace zs
