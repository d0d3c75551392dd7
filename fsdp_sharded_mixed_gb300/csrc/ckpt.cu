// ckpt.cu — block checksums of checkpoint data on the device.
//
// A checkpoint shard of device-resident state is hashed where it lives before
// it is copied to the host (save) and again after the file's bytes are copied
// back (load), so the check covers the host link as well as the file. One
// CTA hashes one block (1 MiB in the file format): 16-byte loads, four in
// flight per thread, the word terms of block_hash.h summed per thread, then
// over the CTA. Bound: HBM, one read of each byte; the mixing is integer
// work well under the read time.
#include <cuda_runtime.h>
#include <stdint.h>

#include "block_hash.h"
#include "zs_internal.h"

namespace zs {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint64_t terms16(uint4 v, uint64_t c) {
  const uint64_t lo = (uint64_t)v.x | ((uint64_t)v.y << 32);
  const uint64_t hi = (uint64_t)v.z | ((uint64_t)v.w << 32);
  return hash_word(lo, c) + hash_word(hi, c + 1);
}

// Block j of the launch: bytes [j*block_bytes, min((j+1)*block_bytes, bytes))
// of `data` (16-byte aligned), which is block first_block + j of its array.
__global__ void __launch_bounds__(kThreads) block_hash_kernel(const unsigned char* data,
                                                              int64_t bytes, int64_t first_block,
                                                              int64_t block_bytes,
                                                              uint32_t array_id, uint64_t* out) {
  const int64_t j = blockIdx.x;
  const int64_t b0 = j * block_bytes;
  const int64_t len = bytes - b0 < block_bytes ? bytes - b0 : block_bytes;
  const unsigned char* p = data + b0;
  const uint64_t base = hash_base(array_id, first_block + j, block_bytes);
  const int64_t nv = len / 16;
  constexpr int U = 4;
  uint64_t acc = 0;
  for (int64_t i0 = 0; i0 < nv; i0 += (int64_t)kThreads * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * kThreads + threadIdx.x;
      if (i < nv) v[u] = ld_stream(p + 16 * i);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * kThreads + threadIdx.x;
      if (i < nv) acc += terms16(v[u], base + 2 * (uint64_t)i + 1);
    }
  }
  if (threadIdx.x == 0) {
    // The last len % 16 bytes: one or two words, the last zero-padded.
    for (int64_t w = nv * 16; w < len; w += 8) {
      uint64_t word = 0;
      for (int k = 0; k < 8 && w + k < len; ++k) word |= (uint64_t)p[w + k] << (8 * k);
      acc += hash_word(word, base + (uint64_t)(w / 8) + 1);
    }
  }
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, off);
  __shared__ uint64_t warp_sum[kThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t s = hash_seed(len, array_id);
    for (int w = 0; w < kThreads / 32; ++w) s += warp_sum[w];
    out[j] = s;
  }
}

}  // namespace

cudaError_t launch_block_hash(const void* data, int64_t bytes, int64_t first_block,
                              int64_t block_bytes, uint32_t array_id, uint64_t* out,
                              cudaStream_t stream) {
  if (bytes <= 0) return cudaSuccess;
  const int64_t blocks = (bytes + block_bytes - 1) / block_bytes;
  block_hash_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(
      static_cast<const unsigned char*>(data), bytes, first_block, block_bytes, array_id, out);
  return cudaGetLastError();
}

}  // namespace zs
