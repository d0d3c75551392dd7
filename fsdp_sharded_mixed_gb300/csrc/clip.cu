// clip.cu — global-norm gradient clipping for the sharded step, and the
// non-finite decision every rank shares.
//
// "从 Data Parallel 到 ZeRO/FSDP", "Gradient Accumulation 会改变生命周期": a
// sharded step has to settle whether clipping uses the global norm or the
// local shard's, and whether an overflow is decided by all ranks alike. Here:
// the global L2 norm of the reduced (mean) gradient. Each rank sums the
// squares of its shard's mean gradient (grad_sqnorm_kernel); the N partial
// sums are added in rank order, the square root taken and the coefficient
// min(1, max_norm / (norm + 1e-6)) formed in double and rounded to fp32
// (clip_coef_kernel, the scalar AllReduce of a real system emulated on one
// GPU); the step multiplies the mean gradient by it, and a non-finite norm
// makes the step leave every buffer untouched.
//
// The norm pass reads the N slices once (g*N bytes per element); for a step
// that ends gradient accumulation it takes the norm of the gradient that step
// sees, (accum + mean) * (1/G), and also reads the accumulator (4 more bytes). Squares are
// formed in fp32 with their exact rounding residue (an FMA), summed per
// 16-element group with a compensated (two-sum) fp32 accumulator, and folded
// into a per-thread double; double work is one add per group, because GB300's
// fp64 rate is far below its fp32 rate. A batch of slices is loaded before it
// is summed, so its loads are in flight together. The grid is a fixed 1216
// blocks (8 per SM of a 152-SM GB300: whole waves at 1, 2, 4 or 8 resident
// blocks per SM); each block's partial goes to scratch memory and the last
// block to finish adds the partials in block order: the result does not depend
// on timing or on the GPU, and is the same on every run.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "bounds.cuh"
#include "overlap.cuh"
#include "zs_internal.h"

namespace zs {
namespace {

constexpr int kThreads = 256;
constexpr int kGW = 16;

template <int MAXN>
struct NormArgs {
  const void* grads[MAXN];
  int64_t lo, hi;
  int world;
  float invN;
  double* partials;        // [kNormPartials]
  unsigned int* ticket;    // zero on entry; the last block resets it
  double* out;
  int64_t win_lo, win_hi;  // checked build: the elements any read may touch
  unsigned int* err;       // checked build: the device error word
  const float* accum;      // ACC: fp32 sum of the earlier micro-steps' mean gradients
  float invG;              // ACC: fp32(1/G)
  bool top_down;           // walk the range from its top (see the kernel)
};

__device__ __forceinline__ void ld32_nc(const void* p, uint32_t* r) {
  asm("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "l"(p));
}

// Compensated accumulation of g*g: s + c carries the group's sum with the
// rounding errors of the squares (exact residues) and of the additions.
__device__ __forceinline__ void acc_square(float g, float& s, float& c) {
  const float hi = __fmul_rn(g, g);
  const float lo = __fmaf_rn(g, g, -hi);
  const float t = __fadd_rn(s, hi);
  const float bv = __fsub_rn(t, s);
  const float av = __fsub_rn(t, bv);
  const float err = __fadd_rn(__fsub_rn(s, av), __fsub_rn(hi, bv));
  s = t;
  c = __fadd_rn(c, __fadd_rn(err, lo));
}

// The gradient the step sees at element i: the mean of the slices; with ACC,
// the micro-batch average (accum + mean) * (1/G).
template <bool BF16G, bool ACC, int MAXN>
__device__ __forceinline__ float mean_grad(const NormArgs<MAXN>& a, int64_t i) {
  if (!within(i, i + 1, a.win_lo, a.win_hi, a.err)) return 0.0f;
  float acc = 0.0f;
  for (int j = 0; j < a.world; ++j) {
    const float x = BF16G ? __uint_as_float(
                                (uint32_t) static_cast<const uint16_t*>(a.grads[j])[i] << 16)
                          : static_cast<const float*>(a.grads[j])[i];
    acc = __fadd_rn(acc, x);
  }
  const float mean = __fmul_rn(acc, a.invN);
  return ACC ? __fmul_rn(__fadd_rn(a.accum[i], mean), a.invG) : mean;
}

// VEC: 16-element groups with 32-byte loads (all slices, and with ACC the
// accumulator, 32-byte aligned); otherwise element by element. ACC: the norm
// of the accumulated step's gradient (accum + mean) * (1/G). A pass that reads
// under 1 GiB walks the range from the top down: the clipped step that follows
// reads the same slices (and accumulator) from the bottom up, so it starts on
// the ones this pass read last, still in L2 (GPT-2-small, N = 8, in place in
// the clip pipeline on GB300: 145.7 against 147.5 us per optimizer step).
// Larger passes go bottom up: there the reuse is a fraction of a percent, and
// the top-down walk measured up to 2 % slower on the Llama-7B shard.
template <bool BF16G, bool VEC, int MAXN, bool ACC>
__global__ void __launch_bounds__(kThreads, 2) grad_sqnorm_kernel(const __grid_constant__ NormArgs<MAXN> a) {
  overlap_wait();
  const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  double sum = 0.0;
  int64_t g0 = 0, g1 = 0;
  if (VEC) {
    g0 = (a.lo + kGW - 1) / kGW;
    g1 = a.hi / kGW;
  }
  if (g0 >= g1) {
    for (int64_t q = tid; q < a.hi - a.lo; q += stride) {
      const int64_t i = a.top_down ? a.hi - 1 - q : a.lo + q;
      const float g = mean_grad<BF16G, ACC>(a, i);
      float s = 0.0f, c = 0.0f;
      acc_square(g, s, c);
      sum += (double)s + (double)c;
    }
  } else {
    const int64_t head = g0 * kGW - a.lo, tail = a.hi - g1 * kGW;
    if (tid < head + tail) {
      const int64_t i = tid < head ? a.lo + tid : g1 * kGW + (tid - head);
      const float g = mean_grad<BF16G, ACC>(a, i);
      float s = 0.0f, c = 0.0f;
      acc_square(g, s, c);
      sum += (double)s + (double)c;
    }
    constexpr int W = BF16G ? kGW / 2 : kGW;          // 32-bit words per slice per group
    constexpr int KB = 64 / W;                        // slices loaded back to back
    constexpr int kStride = BF16G ? 2 * kGW : 4 * kGW;
    for (int64_t q = tid; q < g1 - g0; q += stride) {
      const int64_t g = a.top_down ? g1 - 1 - q : g0 + q;
      if (!within(kGW * g, kGW * g + kGW, a.win_lo, a.win_hi, a.err)) continue;
      float acc[kGW];
#pragma unroll
      for (int k = 0; k < kGW; ++k) acc[k] = 0.0f;
      for (int j0 = 0; j0 < a.world; j0 += KB) {
        uint32_t raw[KB][W];
#pragma unroll
        for (int b = 0; b < KB; ++b) {
          if (j0 + b < a.world) {
            const unsigned char* base =
                static_cast<const unsigned char*>(a.grads[j0 + b]) + g * kStride;
            ld32_nc(base, raw[b]);
            if (!BF16G) ld32_nc(base + 32, raw[b] + 8);
          }
        }
#pragma unroll
        for (int b = 0; b < KB; ++b) {
          if (j0 + b < a.world) {
#pragma unroll
            for (int k = 0; k < W; ++k) {
              if (BF16G) {
                acc[2 * k] = __fadd_rn(acc[2 * k], __uint_as_float(raw[b][k] << 16));
                acc[2 * k + 1] = __fadd_rn(acc[2 * k + 1], __uint_as_float(raw[b][k] & 0xFFFF0000u));
              } else {
                acc[k] = __fadd_rn(acc[k], __uint_as_float(raw[b][k]));
              }
            }
          }
        }
      }
      float prev[ACC ? kGW : 1];
      if constexpr (ACC) {
        const float* ap = a.accum + kGW * g;
        ld32_nc(ap, reinterpret_cast<uint32_t*>(prev));
        ld32_nc(ap + 8, reinterpret_cast<uint32_t*>(prev) + 8);
      }
      float s = 0.0f, c = 0.0f;
#pragma unroll
      for (int k = 0; k < kGW; ++k) {
        const float mean = __fmul_rn(acc[k], a.invN);
        acc_square(ACC ? __fmul_rn(__fadd_rn(prev[k], mean), a.invG) : mean, s, c);
      }
      sum += (double)s + (double)c;
    }
  }
  // Block sum in a fixed order: warp shuffle tree, then warp 0 over the warps.
  __shared__ double warp_sums[kThreads / 32];
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_down_sync(0xFFFFFFFFu, sum, off);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = sum;
  __syncthreads();
  __shared__ bool last;
  if (threadIdx.x == 0) {
    double b = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) b += warp_sums[w];
    if (within(blockIdx.x, blockIdx.x + 1, 0, kNormPartials, a.err)) a.partials[blockIdx.x] = b;
    __threadfence();
    last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  // The last block adds the partials in a fixed order: thread k the partials
  // k, k + 256, ... (all its loads in flight at once, read at L2 where the
  // other blocks' fenced stores are), then the same shuffle tree and warp
  // order as the block sums above.
  __threadfence();
  double t = 0.0;
  double p[(kNormPartials + kThreads - 1) / kThreads];
#pragma unroll
  for (int k = 0; k < (kNormPartials + kThreads - 1) / kThreads; ++k) {
    const unsigned int b = threadIdx.x + k * kThreads;
    p[k] = b < gridDim.x ? __ldcg(a.partials + b) : 0.0;
  }
#pragma unroll
  for (int k = 0; k < (kNormPartials + kThreads - 1) / kThreads; ++k) t += p[k];
  for (int off = 16; off > 0; off >>= 1) t += __shfl_down_sync(0xFFFFFFFFu, t, off);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    double total = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) total += warp_sums[w];
    *a.out = total;
    *a.ticket = 0u;
  }
}

__global__ void clip_coef_kernel(const double* rank_sqnorms, int n, double max_norm, float* coef,
                                 int32_t* nonfinite) {
  overlap_wait();
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  double total = 0.0;
  for (int r = 0; r < n; ++r) total = total + rank_sqnorms[r];
  const double norm = sqrt(total);
  const bool bad = !isfinite(norm);
  const double c = max_norm / (norm + 1e-6);
  *nonfinite = bad ? 1 : 0;
  *coef = bad ? 1.0f : (float)(c < 1.0 ? c : 1.0);
}


template <bool BF16G, bool VEC, int MAXN, bool ACC>
cudaError_t launch_norm(const NormLaunch& in, cudaStream_t stream) {
  NormArgs<MAXN> a;
  for (int j = 0; j < MAXN; ++j) a.grads[j] = (in.grads && j < in.world) ? in.grads[j] : nullptr;
  a.lo = in.lo;
  a.hi = in.hi;
  a.world = in.world;
  a.invN = in.invN;
  a.partials = in.partials;
  a.ticket = in.ticket;
  a.out = in.out;
  a.win_lo = in.win.lo;
  a.win_hi = in.win.hi;
  a.err = ZS_BOUNDS_CHECK ? device_error_word() : nullptr;
  if (ZS_BOUNDS_CHECK && !a.err) return cudaErrorInvalidSymbol;
  a.accum = in.accum;
  a.invG = in.invG;
  const int64_t bytes_per_elem = (int64_t)in.world * (BF16G ? 2 : 4) + (ACC ? 4 : 0);
  a.top_down = (in.hi - in.lo) * bytes_per_elem < (int64_t(1) << 30);
  cudaError_t e = cudaMemsetAsync(in.ticket, 0, sizeof(unsigned int), stream);
  if (e != cudaSuccess) return e;
  return launch_kernel(grad_sqnorm_kernel<BF16G, VEC, MAXN, ACC>, dim3(kNormPartials),
                       dim3(kThreads), 0, stream, a);
}

}  // namespace

template <bool ACC>
cudaError_t dispatch_norm(const NormLaunch& a, cudaStream_t stream) {
  const bool bf16g = a.grad_dtype == ZS_BF16;
  if (a.world <= 16) {
    if (a.vec)
      return bf16g ? launch_norm<true, true, 16, ACC>(a, stream)
                   : launch_norm<false, true, 16, ACC>(a, stream);
    return bf16g ? launch_norm<true, false, 16, ACC>(a, stream)
                 : launch_norm<false, false, 16, ACC>(a, stream);
  }
  if (a.vec)
    return bf16g ? launch_norm<true, true, ZS_MAX_WORLD, ACC>(a, stream)
                 : launch_norm<false, true, ZS_MAX_WORLD, ACC>(a, stream);
  return bf16g ? launch_norm<true, false, ZS_MAX_WORLD, ACC>(a, stream)
               : launch_norm<false, false, ZS_MAX_WORLD, ACC>(a, stream);
}

cudaError_t launch_grad_sqnorm(const NormLaunch& a, cudaStream_t stream) {
  return a.accum ? dispatch_norm<true>(a, stream) : dispatch_norm<false>(a, stream);
}

cudaError_t launch_clip_coef(const double* rank_sqnorms, int n, double max_norm, float* coef,
                             int32_t* nonfinite, cudaStream_t stream) {
  return launch_kernel(clip_coef_kernel, dim3(1), dim3(32), 0, stream, rank_sqnorms, n, max_norm,
                       coef, nonfinite);
}

}  // namespace zs

// ---- The norm pass without caller scratch ------------------------------------
// For callers that cannot allocate device memory, the scratch of one norm pass
// (the 1216 block partials and the ticket word) also exists as a file-scope
// device array. Every GPU that loads this library holds these 9984 bytes until
// the process exits. All calls share it, so calls that overlap on the GPU
// race; the ticket is cleared before each launch and the partials are written
// before they are read, so nothing of an earlier call leaks into a later one.
namespace zs {

static __device__ __align__(256) unsigned char g_norm_scratch[kNoAllocScratchBytes];

cudaError_t launch_grad_sqnorm_noalloc(const NormLaunch& in, cudaStream_t stream) {
  // The array's device address, looked up once per device with that device
  // current (the first call on a device does this set-up).
  static std::mutex mu;
  static void* addr_by_dev[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!addr_by_dev[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_norm_scratch);
      if (e != cudaSuccess) return e;
      addr_by_dev[dev] = p;
    }
    base = addr_by_dev[dev];
  }
  NormLaunch a = in;
  a.partials = static_cast<double*>(base);
  a.ticket = reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(base) + kNormTicketOffset);
  return launch_grad_sqnorm(a, stream);
}

}  // namespace zs
