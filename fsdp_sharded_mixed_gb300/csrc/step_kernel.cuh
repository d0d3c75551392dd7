// step_kernel.cuh — the fused shard-step kernel templates (loads and stores,
// conversions, the AdamW update, the per-group and per-element paths, launch
// and dispatch), shared by shard_step.cu (the step) and accum.cu (the last
// micro-step of gradient accumulation, ACC = true). Included by .cu files of
// this library only; everything here has internal linkage.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "zs_internal.h"

namespace zs {
namespace {

constexpr int kThreads = 256;

enum ParamKind { kParamBf16 = 0, kParamFp32 = 1, kParamFp24 = 2 };

template <int MAXN>
struct StepArgs {
  const void* grads[MAXN];
  float* master;
  float* m;
  float* v;
  unsigned char* slot;
  int64_t lo, hi;
  int world;
  const float* coef;    // clip coefficient (device), or NULL
  const int32_t* skip;  // shared non-finite decision (device), or NULL
  const float* accum;   // ACC: fp32 sum of the earlier micro-steps' mean gradients
  float invG;           // ACC: fp32(1/G), G micro-steps per optimizer step
  StepScalars s;
};

// ---- global loads and stores -----------------------------------------------
// Gradient slices are read-only for the kernel's lifetime and read once:
// non-coherent path, no L1 allocation. States are read then overwritten by the
// same thread, so they take the coherent path.
__device__ __forceinline__ void ld16_nc(const void* p, uint32_t* r) {
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "l"(p));
}
__device__ __forceinline__ void ld32_nc(const void* p, uint32_t* r) {
  asm("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "l"(p));
}
__device__ __forceinline__ void ld16_f(const float* p, float* r) {
  asm("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3])
      : "l"(p));
}
__device__ __forceinline__ void ld32_f(const float* p, float* r) {
  asm("ld.global.L1::no_allocate.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]),
        "=f"(r[7])
      : "l"(p));
}
__device__ __forceinline__ void st16_u(void* p, const uint32_t* w) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3])
               : "memory");
}
__device__ __forceinline__ void st32_u(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void st8_u(void* p, const uint32_t* w) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(w[0]), "r"(w[1]) : "memory");
}
__device__ __forceinline__ void st16_f(float* p, const float* x) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(x[0]), "f"(x[1]),
               "f"(x[2]), "f"(x[3])
               : "memory");
}
__device__ __forceinline__ void st32_f(float* p, const float* x) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(x[0]),
               "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7])
               : "memory");
}

// GW consecutive fp32 values (a group's worth of one state array).
template <int GW>
__device__ __forceinline__ void load_state(const float* p, float* x) {
  if constexpr (GW == 16) {
    ld32_f(p, x);
    ld32_f(p + 8, x + 8);
  } else {
    ld16_f(p, x);
    ld16_f(p + 4, x + 4);
  }
}
template <int GW>
__device__ __forceinline__ void store_state(float* p, const float* x) {
  if constexpr (GW == 16) {
    st32_f(p, x);
    st32_f(p + 8, x + 8);
  } else {
    st16_f(p, x);
    st16_f(p + 4, x + 4);
  }
}
// GW gradient values of one slice as raw words: GW/2 words (bf16) or GW (fp32).
template <int GW, bool BF16G>
__device__ __forceinline__ void load_grad(const void* p, uint32_t* w) {
  if constexpr (BF16G) {
    if constexpr (GW == 16) ld32_nc(p, w);
    else ld16_nc(p, w);
  } else {
    const unsigned char* b = static_cast<const unsigned char*>(p);
    if constexpr (GW == 16) {
      ld32_nc(b, w);
      ld32_nc(b + 32, w + 8);
    } else {
      ld16_nc(b, w);
      ld16_nc(b + 16, w + 4);
    }
  }
}

// ---- conversions -------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t to_bf16(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}
// fp32 -> the 3-byte float (top 24 bits), round to nearest even on the 8
// dropped bits; a NaN stays a (quiet) NaN; the carry of the rounding moves
// into the exponent, so overflow reaches infinity.
__device__ __forceinline__ uint32_t to_fp24(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (b >> 8) | 0x4000u;
  uint32_t keep = b >> 8, rest = b & 0xFFu;
  keep += (rest > 0x80u || (rest == 0x80u && (keep & 1u))) ? 1u : 0u;
  return keep;
}

// ---- the update ----------------------------------------------------------------
// Adam moments with bias correction and the lr-scaled decoupled decay, one
// rounded fp32 operation per step.
__device__ __forceinline__ void adamw(const StepScalars& s, float g, float& p, float& m,
                                      float& v) {
  m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
  v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(__fmul_rn(s.omb2, g), g));
  const float m_hat = __fdiv_rn(m, s.bc1);
  const float v_hat = __fdiv_rn(v, s.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), s.eps);
  const float u = __fdiv_rn(m_hat, denom);
  p = __fsub_rn(__fmul_rn(p, s.decay), __fmul_rn(s.lr, u));
}

// ---- one group of GW elements --------------------------------------------------
// acc[k] = (((0 + x_0) + x_1) + ...) over the slices, j ascending. The slices
// are loaded a batch at a time so that a batch's loads are all in flight
// together (32 words of gradient per thread; a batch of 4 bf16 slices at
// GW = 16). N is a runtime value: on GB300 this measured faster than copies of
// the kernel with N fixed at compile time (1.015 vs 0.977 of the copy
// bandwidth on the Llama-7B shard, 1.009 vs 0.938 on Qwen2.5-3B).
template <int GW, bool BF16G, int MAXN>
__device__ __forceinline__ void reduce_group(const StepArgs<MAXN>& a, int64_t g, float* acc) {
  constexpr int W = BF16G ? GW / 2 : GW;            // 32-bit words per slice per group
  constexpr int KB = 32 / W >= 1 ? 32 / W : 1;      // slices per batch
  constexpr int kStride = BF16G ? 2 * GW : 4 * GW;  // bytes per slice per group
  const int n = a.world;
#pragma unroll
  for (int k = 0; k < GW; ++k) acc[k] = 0.0f;
#pragma unroll 1
  for (int j0 = 0; j0 < n; j0 += KB) {
    uint32_t raw[KB][W];
#pragma unroll
    for (int b = 0; b < KB; ++b)
      if (j0 + b < n)
        load_grad<GW, BF16G>(static_cast<const unsigned char*>(a.grads[j0 + b]) + g * kStride,
                             raw[b]);
#pragma unroll
    for (int b = 0; b < KB; ++b) {
      if (j0 + b < n) {
        if constexpr (BF16G) {
#pragma unroll
          for (int k = 0; k < W; ++k) {
            acc[2 * k] = __fadd_rn(acc[2 * k], bf16_lo(raw[b][k]));
            acc[2 * k + 1] = __fadd_rn(acc[2 * k + 1], bf16_hi(raw[b][k]));
          }
        } else {
#pragma unroll
          for (int k = 0; k < W; ++k) acc[k] = __fadd_rn(acc[k], __uint_as_float(raw[b][k]));
        }
      }
    }
  }
}

template <int GW, int PD>
__device__ __forceinline__ void store_params(unsigned char* slot, int64_t g, const float* p) {
  if constexpr (PD == kParamBf16) {
    uint32_t w[GW / 2];
#pragma unroll
    for (int k = 0; k < GW / 2; ++k) w[k] = pack_bf16x2(p[2 * k], p[2 * k + 1]);
    if constexpr (GW == 16) st32_u(slot + 32 * g, w);
    else st16_u(slot + 16 * g, w);
  } else if constexpr (PD == kParamFp32) {
    store_state<GW>(reinterpret_cast<float*>(slot) + GW * g, p);
  } else {
    // Each run of 8 values is 24 bytes = six little-endian words.
    unsigned char* d = slot + 3 * GW * g;
#pragma unroll
    for (int r = 0; r < GW / 8; ++r) {
      uint32_t q[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) q[k] = to_fp24(p[8 * r + k]);
      const uint32_t w[6] = {q[0] | (q[1] << 24), (q[1] >> 8) | (q[2] << 16),
                             (q[2] >> 16) | (q[3] << 8), q[4] | (q[5] << 24),
                             (q[5] >> 8) | (q[6] << 16), (q[6] >> 16) | (q[7] << 8)};
      if constexpr (GW == 16) {
        // 48 bytes per group from a 16-byte aligned start: 16 + 8 | 8 + 16.
        if (r == 0) {
          st16_u(d, w);
          st8_u(d + 16, w + 4);
        } else {
          st8_u(d + 24, w);
          st16_u(d + 32, w + 2);
        }
      } else {
        st8_u(d, w);
        st8_u(d + 8, w + 2);
        st8_u(d + 16, w + 4);
      }
    }
  }
}

// The gradient the update sees: the mean of the slices; with ACC, the
// micro-step average ((sum of the earlier means) + this mean) * (1/G); times
// the clip coefficient when clipping.
template <bool ACC>
__device__ __forceinline__ float step_grad(float acc, float prev, float invN, float invG,
                                           bool clip, float coef) {
  float g = __fmul_rn(acc, invN);
  if constexpr (ACC) g = __fmul_rn(__fadd_rn(prev, g), invG);
  return clip ? __fmul_rn(g, coef) : g;
}

template <int GW, bool BF16G, int PD, int MAXN, bool ACC>
__device__ __forceinline__ void process_group(const StepArgs<MAXN>& a, int64_t g, bool clip,
                                              float coef) {
  float p[GW], m[GW], v[GW], acc[GW], prev[ACC ? GW : 1];
  load_state<GW>(a.master + GW * g, p);
  load_state<GW>(a.m + GW * g, m);
  load_state<GW>(a.v + GW * g, v);
  if constexpr (ACC) load_state<GW>(a.accum + GW * g, prev);
  reduce_group<GW, BF16G>(a, g, acc);
#pragma unroll
  for (int k = 0; k < GW; ++k)
    adamw(a.s, step_grad<ACC>(acc[k], ACC ? prev[k] : 0.0f, a.s.invN, a.invG, clip, coef),
          p[k], m[k], v[k]);
  store_state<GW>(a.master + GW * g, p);
  store_state<GW>(a.m + GW * g, m);
  store_state<GW>(a.v + GW * g, v);
  store_params<GW, PD>(a.slot, g, p);
}

// One element, for the ragged head/tail and unaligned slots.
template <bool BF16G, int PD, int MAXN, bool ACC>
__device__ __forceinline__ void process_element(const StepArgs<MAXN>& a, int64_t i, bool clip,
                                                float coef) {
  float acc = 0.0f;
  for (int j = 0; j < a.world; ++j) {
    const float x = BF16G ? __uint_as_float(
                                (uint32_t) static_cast<const uint16_t*>(a.grads[j])[i] << 16)
                          : static_cast<const float*>(a.grads[j])[i];
    acc = __fadd_rn(acc, x);
  }
  float p = a.master[i], m = a.m[i], v = a.v[i];
  adamw(a.s, step_grad<ACC>(acc, ACC ? a.accum[i] : 0.0f, a.s.invN, a.invG, clip, coef), p, m,
        v);
  a.master[i] = p;
  a.m[i] = m;
  a.v[i] = v;
  if constexpr (PD == kParamBf16) {
    reinterpret_cast<uint16_t*>(a.slot)[i] = to_bf16(p);
  } else if constexpr (PD == kParamFp32) {
    reinterpret_cast<float*>(a.slot)[i] = p;
  } else {
    const uint32_t q = to_fp24(p);
    unsigned char* d = a.slot + 3 * i;
    d[0] = (unsigned char)(q & 0xFFu);
    d[1] = (unsigned char)((q >> 8) & 0xFFu);
    d[2] = (unsigned char)((q >> 16) & 0xFFu);
  }
}

// GW = 0: every element one by one. GW = 8 or 16: whole groups vectorised.
template <int GW, bool BF16G, int PD, int MAXN, bool ACC>
__global__ void __launch_bounds__(kThreads, 2)
    shard_step_kernel(const __grid_constant__ StepArgs<MAXN> a) {
  if (a.skip && *a.skip) return;  // the ranks' shared non-finite decision
  const bool clip = a.coef != nullptr;
  const float coef = clip ? *a.coef : 1.0f;
  const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  int64_t g0 = 0, g1 = 0;
  if constexpr (GW > 0) {
    g0 = (a.lo + GW - 1) / GW;
    g1 = a.hi / GW;
  }
  if (g0 >= g1) {  // no whole group: everything is ragged
    for (int64_t i = a.lo + tid; i < a.hi; i += stride)
      process_element<BF16G, PD, MAXN, ACC>(a, i, clip, coef);
    return;
  }
  if constexpr (GW > 0) {
    const int64_t head = g0 * GW - a.lo, tail = a.hi - g1 * GW;
    if (tid < head) process_element<BF16G, PD, MAXN, ACC>(a, a.lo + tid, clip, coef);
    else if (tid < head + tail)
      process_element<BF16G, PD, MAXN, ACC>(a, g1 * GW + (tid - head), clip, coef);
    for (int64_t g = g0 + tid; g < g1; g += stride)
      process_group<GW, BF16G, PD, MAXN, ACC>(a, g, clip, coef);
  }
}

template <int GW, bool BF16G, int PD, int MAXN, bool ACC>
cudaError_t launch_one(const ShardStepLaunch& in, cudaStream_t stream) {
  // Resident blocks on the whole GPU for this instantiation, per device; the
  // grid is twice that, so the tail of one wave overlaps the next.
  static int max_blocks_by_dev[64];
  auto kernel = shard_step_kernel<GW, BF16G, PD, MAXN, ACC>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int& max_blocks = max_blocks_by_dev[dev & 63];
  if (max_blocks == 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
    if (e != cudaSuccess) return e;
    max_blocks = 2 * sms * (per_sm > 0 ? per_sm : 1);
  }
  StepArgs<MAXN> a;
  for (int j = 0; j < in.world; ++j) a.grads[j] = in.grads[j];
  for (int j = in.world; j < MAXN; ++j) a.grads[j] = nullptr;
  a.master = in.master;
  a.m = in.m;
  a.v = in.v;
  a.slot = in.slot;
  a.lo = in.lo;
  a.hi = in.hi;
  a.world = in.world;
  a.coef = in.coef;
  a.skip = in.skip;
  a.accum = in.accum;
  a.invG = in.invG;
  a.s = in.s;
  const int64_t units = GW > 0 ? (in.hi - in.lo) / GW + 2 : (in.hi - in.lo);
  int64_t blocks = (units + kThreads - 1) / kThreads;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <bool BF16G, int PD, bool ACC>
cudaError_t dispatch(const ShardStepLaunch& a, cudaStream_t stream) {
  if (a.vec_width == 16) {
    if (a.world <= 16) return launch_one<16, BF16G, PD, 16, ACC>(a, stream);
    return launch_one<16, BF16G, PD, ZS_MAX_WORLD, ACC>(a, stream);
  }
  if (a.vec_width == 8) return launch_one<8, BF16G, PD, ZS_MAX_WORLD, ACC>(a, stream);
  return launch_one<0, BF16G, PD, ZS_MAX_WORLD, ACC>(a, stream);
}

// The step with or without the micro-step accumulator, every dtype pair.
template <bool ACC>
cudaError_t launch_step_kernel(const ShardStepLaunch& a, cudaStream_t stream) {
  const bool bf16g = a.grad_dtype == ZS_BF16;
  switch (a.param_dtype) {
    case ZS_BF16:
      return bf16g ? dispatch<true, kParamBf16, ACC>(a, stream)
                   : dispatch<false, kParamBf16, ACC>(a, stream);
    case ZS_FP32:
      return bf16g ? dispatch<true, kParamFp32, ACC>(a, stream)
                   : dispatch<false, kParamFp32, ACC>(a, stream);
    case ZS_FP24:
      return bf16g ? dispatch<true, kParamFp24, ACC>(a, stream)
                   : dispatch<false, kParamFp24, ACC>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

}  // namespace zs
