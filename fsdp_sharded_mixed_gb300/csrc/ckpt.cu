// ckpt.cu — block checksums of checkpoint data on the device.
//
// A checkpoint shard of device-resident state is hashed where it lives before
// it is copied to the host (save) and again after the file's bytes are copied
// back (load), so the check covers the host link as well as the file. A
// block (1 MiB in the file format) is hashed by one or more CTAs, as many as
// it takes to give a launch 8 CTAs per SM: 16-byte loads, four in flight per
// thread, the word terms of block_hash.h summed per thread, then over the
// CTA. Bound: HBM, one read of each byte; the mixing is integer work well
// under the read time.
#include <cuda_runtime.h>
#include <stdint.h>

#include "block_hash.h"
#include "bounds.cuh"
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

// Block j of the launch is bytes [j*block_bytes, min((j+1)*block_bytes,
// bytes)) of `data` (16-byte aligned), block first_block + j of its array.
// It is cut into `parts` equal slices (a multiple of 16 bytes each), one per
// CTA, so that a launch over few blocks still spreads over every SM: CTA
// (j, p) writes the sum of its slice's word terms, plus the block's seed term
// when p = 0, to out[j*parts + p]; the block's checksum is the sum of its
// parts (mod 2^64, in any order).
__global__ void __launch_bounds__(kThreads) block_hash_kernel(const unsigned char* data,
                                                              int64_t bytes, int64_t first_block,
                                                              int64_t block_bytes,
                                                              uint32_t array_id, int parts,
                                                              uint64_t* out, unsigned int* err) {
  const int64_t j = blockIdx.x / parts;
  const int p = (int)(blockIdx.x % parts);
  const int64_t len = bytes - j * block_bytes < block_bytes ? bytes - j * block_bytes
                                                             : block_bytes;
  const int64_t slice = block_bytes / parts;
  const int64_t s0 = p * slice;
  const int64_t s1 = s0 + slice < len ? s0 + slice : len;
  const unsigned char* blk = data + j * block_bytes;
  // Checked build: the slice lies in its block, and the block in the data.
  const bool ok = within(j * block_bytes, j * block_bytes + len, 0, bytes, err) &&
                  (s0 >= s1 || within(s0, s1, 0, len, err));
  const uint64_t base = hash_base(array_id, first_block + j, block_bytes);
  constexpr int U = 4;
  uint64_t acc = 0;
  if (ok && s0 < s1) {
    // 16-byte vectors i in [v0, v1) of the block (word 2i and 2i + 1).
    const int64_t v0 = s0 / 16, v1 = s1 / 16;
    for (int64_t i0 = v0; i0 < v1; i0 += (int64_t)kThreads * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + u * kThreads + threadIdx.x;
        if (i < v1) v[u] = ld_stream(blk + 16 * i);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + u * kThreads + threadIdx.x;
        if (i < v1) acc += terms16(v[u], base + 2 * (uint64_t)i + 1);
      }
    }
    if (threadIdx.x == 0 && s1 == len) {
      // The block's last len % 16 bytes: one or two words, the last zero-padded.
      for (int64_t w = v1 * 16; w < len; w += 8) {
        uint64_t word = 0;
        for (int k = 0; k < 8 && w + k < len; ++k) word |= (uint64_t)blk[w + k] << (8 * k);
        acc += hash_word(word, base + (uint64_t)(w / 8) + 1);
      }
    }
  }
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, off);
  __shared__ uint64_t warp_sum[kThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0 && within(blockIdx.x, blockIdx.x + 1, 0, (int64_t)gridDim.x, err)) {
    uint64_t sum = p == 0 ? hash_seed(len, array_id) : 0;
    for (int w = 0; w < kThreads / 32; ++w) sum += warp_sum[w];
    out[blockIdx.x] = sum;
  }
}

}  // namespace

cudaError_t launch_block_hash(const void* data, int64_t bytes, int64_t first_block,
                              int64_t block_bytes, uint32_t array_id, int parts, uint64_t* out,
                              cudaStream_t stream) {
  if (bytes <= 0) return cudaSuccess;
  const int64_t blocks = (bytes + block_bytes - 1) / block_bytes;
  unsigned int* err = ZS_BOUNDS_CHECK ? device_error_word() : nullptr;
  if (ZS_BOUNDS_CHECK && !err) return cudaErrorInvalidSymbol;
  block_hash_kernel<<<(unsigned)(blocks * parts), kThreads, 0, stream>>>(
      static_cast<const unsigned char*>(data), bytes, first_block, block_bytes, array_id, parts,
      out, err);
  return cudaGetLastError();
}

int block_hash_parts(int64_t blocks, int64_t block_bytes) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    sms = 152;
  }
  const int64_t target = 8 * (int64_t)sms;  // CTAs: 8 resident per SM
  int parts = 1;
  while (blocks * parts < target && block_bytes / (parts * 2) >= 4096) parts *= 2;
  return parts;
}

}  // namespace zs
