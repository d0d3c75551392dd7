// rows.cu — the FSDP2 gather side for per-parameter Shard(0) parameters.
//
// "FSDP2's parameter lifecycle…", "The parameter lifecycle, one module at a
// time": before a module's forward the parameters are all-gathered and
// materialised in full, afterwards resharded (to 1/N, or with an integer
// reshard_after_forward to a smaller world); "从 Data Parallel 到 ZeRO/FSDP",
// "ZeRO 与 FSDP 的关系": FSDP2 shards every parameter on its own (per-parameter
// DTensor). Under that layout the AllGather output is rank-major (each rank's
// chunks of all the unit's parameters back to back), so the gathered rows must
// be copied out into each parameter's own tensor (zs_unshard), and resharding
// copies a rank's rows back into a local buffer (zs_shard_rows).
//
// Both are one kernel: a list of segments, each a plain copy of a byte run plus
// a zero-filled tail (the padding rows of a chunk). A launch takes up to
// kMaxSegs segments as kernel parameters (no device-side table). The bytes of
// all its segments are cut into 32 KB chunks and the blocks stride over the
// chunks (a binary search over the segments' chunk prefix sums finds a chunk's
// segment), so the load is even however unequal the segments are (a unit mixes
// 1 KB norm rows with 11 MB MLP chunks); each chunk moves with the widest
// access its segment's alignment allows (32 bytes for real layouts). Bound:
// HBM, 2 bytes of traffic per byte copied (read + write) and 1 per zero byte.
#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.cuh"
#include "overlap.cuh"
#include "zs_internal.h"

namespace zs {
namespace {

constexpr int kThreads = 256;
constexpr int64_t kChunk = 32 * 1024;  // bytes of one segment a block copies at a time

// A launch's segments and, for load balance, the prefix sums of their chunk
// counts: chunk c of the launch is chunk c - first[s] of the segment s with
// first[s] <= c < first[s + 1]. A segment's byte run is its copy bytes then
// its zero bytes.
struct SegArgs {
  RowSegment seg[kMaxSegs];
  int64_t first[kMaxSegs + 1];
  int count;
  unsigned int* err;  // checked build: the device error word
};

__device__ __forceinline__ uint4 ld_once(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
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

// 32-byte aligned run: 32-byte loads and stores, 4 loads in flight per thread
// (32 KB per block).
__device__ __forceinline__ void copy_range32(const unsigned char* src, unsigned char* dst,
                                             int64_t b0, int64_t b1) {
  constexpr int U = 4;
  const int n = (int)((b1 - b0) / 32);
  for (int base = 0; base < n; base += kThreads * U) {
    uint32_t r[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kThreads + threadIdx.x;
      if (i < n) ld32_once(src + b0 + 32 * (int64_t)i, r[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kThreads + threadIdx.x;
      if (i < n) st32(dst + b0 + 32 * (int64_t)i, r[u]);
    }
  }
}

// 16-byte aligned run: each thread issues 4 loads before its stores, so a
// block keeps 16 KB in flight.
__device__ __forceinline__ void copy_range16(const unsigned char* src, unsigned char* dst,
                                             int64_t b0, int64_t b1) {
  constexpr int U = 4;
  const uint4* s = reinterpret_cast<const uint4*>(src + b0);
  uint4* d = reinterpret_cast<uint4*>(dst + b0);
  const int n = (int)((b1 - b0) / 16);
  for (int base = 0; base < n; base += kThreads * U) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kThreads + threadIdx.x;
      if (i < n) r[u] = ld_once(s + i);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kThreads + threadIdx.x;
      if (i < n) d[i] = r[u];
    }
  }
}

template <typename T>
__device__ __forceinline__ void copy_range(const unsigned char* src, unsigned char* dst,
                                           int64_t b0, int64_t b1) {
  const T* s = reinterpret_cast<const T*>(src + b0);
  T* d = reinterpret_cast<T*>(dst + b0);
  const int64_t n = (b1 - b0) / (int64_t)sizeof(T);
  for (int64_t i = threadIdx.x; i < n; i += kThreads) d[i] = s[i];
}

template <typename T>
__device__ __forceinline__ void zero_range(unsigned char* dst, int64_t b0, int64_t b1) {
  T* d = reinterpret_cast<T*>(dst + b0);
  const int64_t n = (b1 - b0) / (int64_t)sizeof(T);
  T z;
  memset(&z, 0, sizeof z);
  for (int64_t i = threadIdx.x; i < n; i += kThreads) d[i] = z;
}

__device__ __forceinline__ int unit_of(uintptr_t a) {
  return (a & 31u) == 0   ? 32
         : (a & 15u) == 0 ? 16
         : (a & 7u) == 0  ? 8
         : (a & 3u) == 0  ? 4
         : (a & 1u) == 0  ? 2
                          : 1;
}

__global__ void __launch_bounds__(kThreads) segment_copy_kernel(const __grid_constant__ SegArgs a) {
  overlap_wait();
  const int64_t total = a.first[a.count];
  for (int64_t c = blockIdx.x; c < total; c += gridDim.x) {
    int lo = 0, hi = a.count - 1;  // the segment holding chunk c
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.first[mid] <= c) lo = mid;
      else hi = mid - 1;
    }
    if (!within(lo, lo + 1, 0, a.count, a.err)) continue;
    const RowSegment& s = a.seg[lo];
    const int64_t b0 = (c - a.first[lo]) * kChunk;
    const int64_t len = s.copy_bytes + s.zero_bytes;
    const int64_t b1 = b0 + kChunk < len ? b0 + kChunk : len;
    // Checked build: the chunk lies inside its segment's byte run.
    if (!within(b0, b1, 0, len, a.err)) continue;
    // Copy part [b0, min(b1, copy_bytes)); chunk edges are multiples of kChunk,
    // so the widest unit dividing the segment's base addresses and copy length
    // also divides every chunk edge inside it.
    const int64_t c1 = b1 < s.copy_bytes ? b1 : s.copy_bytes;
    if (b0 < c1 && within(b0, c1, 0, s.copy_bytes, a.err)) {
      const int64_t e = c1 == s.copy_bytes ? s.copy_bytes : kChunk;
      switch (unit_of((uintptr_t)s.src | (uintptr_t)s.dst | (uintptr_t)e)) {
        case 32: copy_range32(s.src, s.dst, b0, c1); break;
        case 16: copy_range16(s.src, s.dst, b0, c1); break;
        case 8: copy_range<uint2>(s.src, s.dst, b0, c1); break;
        case 4: copy_range<uint32_t>(s.src, s.dst, b0, c1); break;
        case 2: copy_range<uint16_t>(s.src, s.dst, b0, c1); break;
        default: copy_range<uint8_t>(s.src, s.dst, b0, c1); break;
      }
      // Odd tail bytes the unit did not cover (only when c1 is the run's end).
      const int u = unit_of((uintptr_t)s.src | (uintptr_t)s.dst | (uintptr_t)e);
      const int64_t done = b0 + (c1 - b0) / u * u;
      for (int64_t i = done + threadIdx.x; i < c1; i += kThreads) s.dst[i] = s.src[i];
    }
    // Zero part [max(b0, copy_bytes), b1).
    const int64_t z0 = b0 > s.copy_bytes ? b0 : s.copy_bytes;
    if (z0 < b1 && within(z0, b1, s.copy_bytes, len, a.err)) {
      // From the first 16-byte boundary at or after z0 to the last one at or
      // before b1: whole 16-byte stores; the bytes around them one by one.
      const int64_t a0 = (int64_t)((((uintptr_t)(s.dst + z0) + 15u) & ~(uintptr_t)15u) -
                                   (uintptr_t)s.dst);
      const int64_t a1 = (int64_t)((((uintptr_t)(s.dst + b1)) & ~(uintptr_t)15u) -
                                   (uintptr_t)s.dst);
      if (a0 < a1) {
        zero_range<uint4>(s.dst, a0, a1);
        for (int64_t i = z0 + threadIdx.x; i < a0; i += kThreads) s.dst[i] = 0;
        for (int64_t i = a1 + threadIdx.x; i < b1; i += kThreads) s.dst[i] = 0;
      } else {
        for (int64_t i = z0 + threadIdx.x; i < b1; i += kThreads) s.dst[i] = 0;
      }
    }
  }
}

}  // namespace

cudaError_t launch_segment_copy(const RowSegment* segs, int n, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  for (int first = 0; first < n; first += kMaxSegs) {
    SegArgs a;
    a.err = ZS_BOUNDS_CHECK ? device_error_word() : nullptr;
    if (ZS_BOUNDS_CHECK && !a.err) return cudaErrorInvalidSymbol;
    a.count = n - first < kMaxSegs ? n - first : kMaxSegs;
    a.first[0] = 0;
    for (int k = 0; k < a.count; ++k) {
      a.seg[k] = segs[first + k];
      const int64_t len = a.seg[k].copy_bytes + a.seg[k].zero_bytes;
      a.first[k + 1] = a.first[k] + (len + kChunk - 1) / kChunk;
    }
    const int64_t total = a.first[a.count];
    if (total == 0) continue;
    // 8 resident blocks per SM; blocks stride over the launch's chunks.
    const int64_t cap = (int64_t)sms * 8;
    const int64_t blocks = total < cap ? total : cap;
    e = launch_kernel(segment_copy_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace zs
