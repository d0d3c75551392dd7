// bounds.cuh — the access checks of the bounds-checked build.
//
// The library's CUDA sources compiled with ZS_BOUNDS_CHECK=1 (libzs_checked.so)
// check, before each global access or bulk copy, that the range of elements or
// bytes it touches lies inside the window its launch declares: the shard
// range [lo, hi) for the step, accumulation and norm kernels; the slot and
// the world's buffer for the gather; the segment for the row copies; the
// block for the checksums. A range outside its window is not accessed, and
// bit value 1 of the device error word is set, which zs_check_device_error
// reports as ZS_ERR_RANGE. No trap, no assert: the context stays usable.
// In the ordinary build (ZS_BOUNDS_CHECK=0) every check is the constant
// true and compiles away.
#pragma once

#include <stdint.h>

#ifndef ZS_BOUNDS_CHECK
#define ZS_BOUNDS_CHECK 0
#endif

namespace zs {

// [a, b) inside [lo, hi)?
__device__ __forceinline__ bool within(int64_t a, int64_t b, int64_t lo, int64_t hi,
                                       unsigned int* err) {
#if ZS_BOUNDS_CHECK
  if (lo <= a && a <= b && b <= hi) return true;
  atomicOr(err, 1u);
  return false;
#else
  (void)a;
  (void)b;
  (void)lo;
  (void)hi;
  (void)err;
  return true;
#endif
}

}  // namespace zs
