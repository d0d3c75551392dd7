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
// kMaxSegs segments as kernel parameters (no device-side table), blockIdx.y
// picks the segment, blocks stride over its bytes with the widest access the
// segment's alignment allows (16 bytes for real layouts). Bound: HBM, 2 bytes of
// traffic per byte copied (read + write) and 1 per zero byte.
#include <cuda_runtime.h>
#include <stdint.h>

#include "zs_internal.h"

namespace zs {
namespace {

constexpr int kThreads = 256;

struct SegArgs {
  RowSegment seg[kMaxSegs];
};

template <typename T>
__device__ __forceinline__ void copy_run(const unsigned char* src, unsigned char* dst,
                                         int64_t bytes, int64_t start, int64_t stride) {
  const T* s = reinterpret_cast<const T*>(src);
  T* d = reinterpret_cast<T*>(dst);
  const int64_t n = bytes / (int64_t)sizeof(T);
  for (int64_t i = start; i < n; i += stride) d[i] = s[i];
}

template <typename T>
__device__ __forceinline__ void zero_run(unsigned char* dst, int64_t bytes, int64_t start,
                                         int64_t stride) {
  T* d = reinterpret_cast<T*>(dst);
  const int64_t n = bytes / (int64_t)sizeof(T);
  T z;
  memset(&z, 0, sizeof z);
  for (int64_t i = start; i < n; i += stride) d[i] = z;
}

__device__ __forceinline__ int unit_of(uintptr_t a) {
  return (a & 15u) == 0 ? 16 : (a & 7u) == 0 ? 8 : (a & 3u) == 0 ? 4 : (a & 1u) == 0 ? 2 : 1;
}

__global__ void __launch_bounds__(kThreads) segment_copy_kernel(const __grid_constant__ SegArgs a) {
  const RowSegment& s = a.seg[blockIdx.y];
  const int64_t start = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  if (s.copy_bytes > 0) {
    switch (unit_of((uintptr_t)s.src | (uintptr_t)s.dst | (uintptr_t)s.copy_bytes)) {
      case 16: copy_run<uint4>(s.src, s.dst, s.copy_bytes, start, stride); break;
      case 8: copy_run<uint2>(s.src, s.dst, s.copy_bytes, start, stride); break;
      case 4: copy_run<uint32_t>(s.src, s.dst, s.copy_bytes, start, stride); break;
      case 2: copy_run<uint16_t>(s.src, s.dst, s.copy_bytes, start, stride); break;
      default: copy_run<uint8_t>(s.src, s.dst, s.copy_bytes, start, stride); break;
    }
  }
  if (s.zero_bytes > 0) {
    unsigned char* z = s.dst + s.copy_bytes;
    switch (unit_of((uintptr_t)z | (uintptr_t)s.zero_bytes)) {
      case 16: zero_run<uint4>(z, s.zero_bytes, start, stride); break;
      case 8: zero_run<uint2>(z, s.zero_bytes, start, stride); break;
      case 4: zero_run<uint32_t>(z, s.zero_bytes, start, stride); break;
      case 2: zero_run<uint16_t>(z, s.zero_bytes, start, stride); break;
      default: zero_run<uint8_t>(z, s.zero_bytes, start, stride); break;
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
    const int count = n - first < kMaxSegs ? n - first : kMaxSegs;
    SegArgs a;
    int64_t longest = 0;
    for (int k = 0; k < count; ++k) {
      a.seg[k] = segs[first + k];
      const int64_t b = a.seg[k].copy_bytes > a.seg[k].zero_bytes ? a.seg[k].copy_bytes
                                                                  : a.seg[k].zero_bytes;
      if (b > longest) longest = b;
    }
    // Enough blocks per segment for its longest run in 16-byte units, and about
    // 8 resident blocks per SM over all the segments of the launch.
    int64_t bx = (longest / 16 + kThreads - 1) / kThreads;
    const int64_t cap = ((int64_t)sms * 8 + count - 1) / count;
    if (bx > cap) bx = cap;
    if (bx < 1) bx = 1;
    segment_copy_kernel<<<dim3((unsigned)bx, (unsigned)count), kThreads, 0, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace zs
