// bulk.cuh — shared-memory staging by bulk asynchronous copies, for the
// library's staged kernels (the step and the norm pass): mbarriers that count
// the bytes of a stage's copies, bounded waits on them, and the
// one-dimensional bulk copy global -> shared. Included by .cu files of this
// library only; everything here has internal linkage.
#pragma once

#include <stdint.h>

namespace zs {
namespace {

// Polls of a bounded wait before it gives up (a stage's copies land in a few
// microseconds; 2^21 polls are far longer than any of them takes).
constexpr uint32_t kWaitPolls = 1u << 21;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}
// Bounded wait for the phase of parity `parity` to complete: at most `polls`
// polls, then the error word's timeout bit (value 2) is set and the caller
// stops.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, unsigned int* err,
                                          uint32_t polls = kWaitPolls) {
  for (uint32_t it = 0; it < polls; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  atomicOr(err, 2u);
  return false;
}
__device__ __forceinline__ void bulk_to_smem(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
}  // namespace
}  // namespace zs
