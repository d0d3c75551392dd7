// block_hash.h — the checksum of a checkpoint block, one definition compiled
// for the host (checkpoint.cpp) and the device (ckpt.cu).
//
// A block is up to block_bytes bytes of one state array (array id 0 master,
// 1 exp_avg, 2 exp_avg_sq). Read it as little-endian 64-bit words, the last
// one zero-padded; word j of block b has the array-wide counter
// c = (array_id << 56) + b * (block_bytes / 8) + j + 1. The block's hash is
//   mix(len * G + array_id) + sum_j mix(word_j + c_j * G)   (mod 2^64)
// with G = 0x9E3779B97F4A7C15 and mix the SplitMix64 output function (Steele,
// Lea and Flood, "Fast splittable pseudorandom number generators", 2014, with
// the constants of its common 64-bit variant). mix is a bijection, so changing
// any one word changes the sum; the counter ties each word to its place, so
// moved words or swapped blocks change it too. The terms are independent, so
// the sum is a parallel reduction in any order.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define ZS_HASH_FN __host__ __device__ __forceinline__
#else
#define ZS_HASH_FN inline
#endif

namespace zs {

constexpr uint64_t kHashGamma = 0x9E3779B97F4A7C15ull;

ZS_HASH_FN uint64_t hash_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

ZS_HASH_FN uint64_t hash_word(uint64_t word, uint64_t counter) {
  return hash_mix(word + counter * kHashGamma);
}

ZS_HASH_FN uint64_t hash_seed(int64_t len, uint32_t array_id) {
  return hash_mix((uint64_t)len * kHashGamma + array_id);
}

// Counter of word 0 of block `block`, minus one.
ZS_HASH_FN uint64_t hash_base(uint32_t array_id, int64_t block, int64_t block_bytes) {
  return ((uint64_t)array_id << 56) + (uint64_t)block * (uint64_t)(block_bytes / 8);
}

}  // namespace zs
