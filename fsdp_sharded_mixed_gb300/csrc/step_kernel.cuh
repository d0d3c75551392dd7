// step_kernel.cuh — the fused shard-step kernel templates (loads and stores,
// conversions, the AdamW update, the per-group and per-element paths, launch
// and dispatch), shared by shard_step.cu (the step) and accum.cu (the last
// micro-step of gradient accumulation, ACC = true). Included by .cu files of
// this library only; everything here has internal linkage.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "bounds.cuh"
#include "bulk.cuh"
#include "overlap.cuh"
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
  int64_t win_lo, win_hi;  // checked build: the elements any access may touch
  unsigned int* err;       // checked build: the device error word
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
  if (!within(GW * g, GW * g + GW, a.win_lo, a.win_hi, a.err)) return;
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
  if (!within(i, i + 1, a.win_lo, a.win_hi, a.err)) return;
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
  overlap_wait();
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

// ---- the staged path ------------------------------------------------------------
// The same step with the N slices and the state tile staged in shared memory
// by bulk asynchronous copies (cp.async.bulk, completion counted on an
// mbarrier): one producer warp keeps the next tile's copies in flight (its
// lanes issue them in parallel: one thread issuing 35 copies of 2 KB per stage
// held N = 32 bf16 slices to 0.89 of the copy bandwidth, 32 lanes 0.98) while
// 16 consumer warps compute the current one from shared memory, so loads and
// arithmetic overlap instead of alternating per thread. A tile is 512 × E
// elements, each consumer thread E of them: E = 4 (2048 elements) where two
// stages of that fit in a block's shared memory, else E = 2 (1024), which
// stages up to 50 bf16 or 25 fp32 slices; a stage is reused once every consumer
// warp has released it. One block per SM and two stages for calls larger than
// twice the L2, two blocks per SM and up to four stages below (staged_shape):
// on GB300 that streams faster than the register-streaming kernel above
// nearly everywhere (the choice is in try_staged). (E = 1 was measured and left out: with 1 KB and 2 KB copies per
// slice it ran at 0.59 and 0.94-0.96 of the copy bandwidth for N = 64 bf16 and
// N = 32 fp32 slices, where the register-streaming kernel runs at 0.98-1.03.)
// Every wait is bounded: a wait that gives up sets the device error word's
// timeout bit (value 2) and the thread stops; the producer waits, bounded,
// for its own copies before the block exits.
constexpr int kStagedWarps = 16;                     // consumer warps
constexpr int kStagedThreads = (kStagedWarps + 1) * 32;
constexpr int kStagedMaxN = 64;
// Elements of a tile with E elements per consumer thread: 2048 or 1024.
__host__ __device__ constexpr int staged_tile(int E) { return kStagedWarps * 32 * E; }
constexpr int kStagedMaxStages = 4;

struct StagedArgs {
  StepArgs<kStagedMaxN> a;
  int64_t t0, t1;      // whole tiles [t0, t1): elements [t0*T, t1*T), T the tile
  int64_t rag_lo[2], rag_hi[2];  // the ragged head and tail, element by element
  int stages;
  uint32_t stage_bytes;
  unsigned int* err;   // the device error word
};

__device__ __forceinline__ void st_u32(void* p, uint32_t w) {
  asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(w) : "memory");
}

// Bytes of one tile of one slice.
template <bool BF16G, int E>
__host__ __device__ constexpr uint32_t tile_grad_bytes() {
  return staged_tile(E) * (BF16G ? 2 : 4);
}

// E consecutive fp32 values from shared memory (aligned to 4E bytes).
template <int E>
__device__ __forceinline__ void lds_f(const float* p, float* x) {
  static_assert(E == 4 || E == 2, "tile widths of 4 or 2 elements per thread");
  if constexpr (E == 4) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    x[0] = q.x;
    x[1] = q.y;
    x[2] = q.z;
    x[3] = q.w;
  } else {
    const float2 q = *reinterpret_cast<const float2*>(p);
    x[0] = q.x;
    x[1] = q.y;
  }
}
// Consumer c's E values of one staged slice tile, added into acc.
template <int E, bool BF16G>
__device__ __forceinline__ void add_slice(const unsigned char* gp, int c, float* acc) {
  if constexpr (BF16G) {
    if constexpr (E == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(gp + c * 8);
      acc[0] = __fadd_rn(acc[0], bf16_lo(w.x));
      acc[1] = __fadd_rn(acc[1], bf16_hi(w.x));
      acc[2] = __fadd_rn(acc[2], bf16_lo(w.y));
      acc[3] = __fadd_rn(acc[3], bf16_hi(w.y));
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(gp + c * 4);
      acc[0] = __fadd_rn(acc[0], bf16_lo(w));
      acc[1] = __fadd_rn(acc[1], bf16_hi(w));
    }
  } else {
    float x[E];
    lds_f<E>(reinterpret_cast<const float*>(gp) + c * E, x);
#pragma unroll
    for (int k = 0; k < E; ++k) acc[k] = __fadd_rn(acc[k], x[k]);
  }
}
// E fp32 values to global memory (aligned to 4E bytes).
template <int E>
__device__ __forceinline__ void stg_f(float* p, const float* x) {
  if constexpr (E == 4) {
    st16_f(p, x);
  } else {
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
  }
}
// The E cast parameters of elements e0 .. e0 + E - 1 into the slot.
template <int E, int PD>
__device__ __forceinline__ void stg_params(unsigned char* slot, int64_t e0, const float* p) {
  if constexpr (PD == kParamBf16) {
    if constexpr (E == 4) {
      const uint32_t w[2] = {pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3])};
      st8_u(slot + 2 * e0, w);
    } else {
      *reinterpret_cast<uint32_t*>(slot + 2 * e0) = pack_bf16x2(p[0], p[1]);
    }
  } else if constexpr (PD == kParamFp32) {
    stg_f<E>(reinterpret_cast<float*>(slot) + e0, p);
  } else {
    unsigned char* d = slot + 3 * e0;
    if constexpr (E == 4) {  // 12 bytes = three little-endian words
      const uint32_t q0 = to_fp24(p[0]), q1 = to_fp24(p[1]), q2 = to_fp24(p[2]),
                     q3 = to_fp24(p[3]);
      st_u32(d, q0 | (q1 << 24));
      st_u32(d + 4, (q1 >> 8) | (q2 << 16));
      st_u32(d + 8, (q2 >> 16) | (q3 << 8));
    } else {  // 6 bytes = three little-endian half-words
      const uint32_t q0 = to_fp24(p[0]), q1 = to_fp24(p[1]);
      uint16_t* h = reinterpret_cast<uint16_t*>(d);
      h[0] = (uint16_t)(q0 & 0xFFFFu);
      h[1] = (uint16_t)((q0 >> 16) | ((q1 & 0xFFu) << 8));
      h[2] = (uint16_t)(q1 >> 8);
    }
  }
}

template <bool BF16G, int PD, bool ACC, int E>
__global__ void __launch_bounds__(kStagedThreads, 2)
    staged_step_kernel(const __grid_constant__ StagedArgs sa) {
  constexpr int T = staged_tile(E);
  const StepArgs<kStagedMaxN>& a = sa.a;
  overlap_wait();
  if (a.skip && *a.skip) return;  // the ranks' shared non-finite decision
  const bool clip = a.coef != nullptr;
  const float coef = clip ? *a.coef : 1.0f;
  extern __shared__ __align__(128) unsigned char smem[];
  const int NS = sa.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * sa.stage_bytes);
  uint64_t* empty = full + NS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = a.world;
  constexpr uint32_t gtile = tile_grad_bytes<BF16G, E>();
  constexpr uint32_t stile = T * 4;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kStagedWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kStagedWarps) {
    // The producer warp: lane 0 waits for a stage to be free and arms it with
    // the tile's byte count; then the warp's lanes issue its N + 3 (+1) bulk
    // copies, copy k by lane k % 32.
    const int ncopies = n + (ACC ? 4 : 3);
    int64_t i = 0;
    for (int64_t t = sa.t0 + blockIdx.x; t < sa.t1; t += gridDim.x, ++i) {
      const int s = (int)(i % NS);
      const uint32_t use = (uint32_t)(i / NS);
      int ok = 1;
      if (lane == 0 && use > 0) ok = mbar_wait(&empty[s], (use - 1) & 1u, sa.err) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      unsigned char* st = smem + (size_t)s * sa.stage_bytes;
      if (!within(t * T, (t + 1) * T, a.win_lo, a.win_hi, sa.err)) {
        if (lane == 0) mbar_expect_tx(&full[s], 0);  // checked build: the stage completes empty
        __syncwarp();
        continue;
      }
      if (lane == 0) mbar_expect_tx(&full[s], sa.stage_bytes);
      __syncwarp();  // the stage is armed before any of its copies is issued
      for (int k = lane; k < ncopies; k += 32) {
        if (k < n) {
          bulk_to_smem(st + k * gtile, static_cast<const unsigned char*>(a.grads[k]) + t * gtile,
                       gtile, &full[s]);
        } else {
          const int q = k - n;
          const float* src = q == 0 ? a.master : q == 1 ? a.m : q == 2 ? a.v : a.accum;
          bulk_to_smem(st + n * gtile + q * stile, src + t * T, stile, &full[s]);
        }
      }
    }
    // Every copy issued has landed before the block may exit.
    if (lane == 0)
      for (int64_t k = i > NS ? i - NS : 0; k < i; ++k)
        mbar_wait(&full[k % NS], (uint32_t)(k / NS) & 1u, sa.err);
    return;
  }

  // The ragged head and tail, one element per consumer thread of the grid.
  const int c = threadIdx.x;
  {
    const int64_t nh = sa.rag_hi[0] - sa.rag_lo[0], nt = sa.rag_hi[1] - sa.rag_lo[1];
    const int64_t consumers = (int64_t)gridDim.x * (kStagedWarps * 32);
    for (int64_t q = (int64_t)blockIdx.x * (kStagedWarps * 32) + c; q < nh + nt; q += consumers)
      process_element<BF16G, PD, kStagedMaxN, ACC>(
          a, q < nh ? sa.rag_lo[0] + q : sa.rag_lo[1] + (q - nh), clip, coef);
  }
  int64_t i = 0;
  for (int64_t t = sa.t0 + blockIdx.x; t < sa.t1; t += gridDim.x, ++i) {
    const int s = (int)(i % NS);
    const uint32_t use = (uint32_t)(i / NS);
    if (!mbar_wait(&full[s], use & 1u, sa.err)) return;
    if (!within(t * T, (t + 1) * T, a.win_lo, a.win_hi, sa.err)) {
      __syncwarp();  // checked build: an empty stage, released untouched
      if (lane == 0) mbar_arrive(&empty[s]);
      continue;
    }
    const unsigned char* st = smem + (size_t)s * sa.stage_bytes;
    float acc[E];
#pragma unroll
    for (int k = 0; k < E; ++k) acc[k] = 0.0f;
#pragma unroll 1
    for (int j = 0; j < n; ++j) add_slice<E, BF16G>(st + j * gtile, c, acc);
    const float* sp = reinterpret_cast<const float*>(st + n * gtile) + c * E;
    float p[E], m[E], v[E], prev[E];
    lds_f<E>(sp, p);
    lds_f<E>(sp + T, m);
    lds_f<E>(sp + 2 * T, v);
    if constexpr (ACC) {
      lds_f<E>(sp + 3 * T, prev);
    } else {
#pragma unroll
      for (int k = 0; k < E; ++k) prev[k] = 0.0f;
    }
    // The stage's next fill is written by the async proxy: order this
    // thread's reads of it before the warp releases the stage.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
    for (int k = 0; k < E; ++k)
      adamw(a.s, step_grad<ACC>(acc[k], prev[k], a.s.invN, a.invG, clip, coef), p[k], m[k],
            v[k]);
    const int64_t e0 = t * T + (int64_t)c * E;
    stg_f<E>(a.master + e0, p);
    stg_f<E>(a.m + e0, m);
    stg_f<E>(a.v + e0, v);
    stg_params<E, PD>(a.slot, e0, p);
  }
}

// The staged path's launch shape. A call whose algorithmic bytes exceed twice
// the L2 (the steps of every named workload and bucket): one block per SM
// holding two stages (the tile being computed and the next one being filled).
// Measured on GB300 against deeper pipelines and two blocks per SM (same
// tiles): the GPT-2-small step (N = 8, 15.5M elements) ran at 1.004 of the
// copy bandwidth with one block of two stages, 0.857 / 0.840 with three / four
// stages, 0.893 with two blocks of two; the Llama-7B shard at 1.042 against
// 0.962 / 0.927 / 0.950; the GPT-2-small bucket calls (1.2M to 14.4M elements)
// at 0.96 against 0.87. Smaller calls, whose data a step back to back with the
// previous one partly finds in L2: two blocks per SM where two stages of each
// fit, with up to four stages (2^22 elements, N = 4 bf16: 1.12 against 0.94;
// 2^20: 0.76 against 0.66). 0 stages = two stages of this tile do not fit.
inline void staged_shape(uint32_t stage_bytes, int smem_per_sm, int smem_per_block, bool small,
                         int* stages, int* blocks_per_sm) {
  if (!small) {
    *blocks_per_sm = 1;
    *stages = 2 * ((int64_t)stage_bytes + 16) <= smem_per_block ? 2 : 0;
    return;
  }
  const int reserve = 1024 + 16 * kStagedMaxStages;  // per-block system use and barriers
  *blocks_per_sm = 2 * (2 * (int64_t)stage_bytes + reserve) <= smem_per_sm ? 2 : 1;
  int64_t budget = smem_per_sm / *blocks_per_sm - reserve;
  if (budget > smem_per_block - 16 * kStagedMaxStages) budget = smem_per_block - 16 * kStagedMaxStages;
  int64_t ns = budget / stage_bytes;
  if (ns > kStagedMaxStages) ns = kStagedMaxStages;
  *stages = ns >= 2 ? (int)ns : 0;
}

template <bool BF16G, int PD, bool ACC, int E>
cudaError_t launch_staged(const ShardStepLaunch& in, uint32_t stage_bytes, int stages,
                          int blocks_per_sm, int sms, int smem_per_sm, cudaStream_t stream) {
  constexpr int T = staged_tile(E);
  auto kernel = staged_step_kernel<BF16G, PD, ACC, E>;
  // One block per SM whatever else is resident when the blocks are placed:
  // with launch overlap they are dispatched while the previous kernel's
  // blocks drain, and two blocks of a small stage would fit on one SM while
  // another SM got none (measured: the Qwen2.5-3B clip pipeline took 6.08 ms
  // instead of 4.81). A block asks for more than half an SM's shared memory.
  size_t smem = (size_t)stages * stage_bytes + 16 * (size_t)stages;
  if (blocks_per_sm == 1 && smem < (size_t)smem_per_sm / 2) smem = (size_t)smem_per_sm / 2;
  // This instantiation's shared-memory opt-in so far, per device; raised
  // under a lock so that concurrent first calls cannot leave it recorded
  // above what the attribute holds.
  static std::atomic<size_t> smem_set_by_dev[64];
  static std::mutex smem_mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (smem > smem_set_by_dev[dev & 63].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(smem_mu);
    if (smem > smem_set_by_dev[dev & 63].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      smem_set_by_dev[dev & 63].store(smem, std::memory_order_release);
    }
  }
  StagedArgs sa;
  for (int j = 0; j < in.world; ++j) sa.a.grads[j] = in.grads[j];
  for (int j = in.world; j < kStagedMaxN; ++j) sa.a.grads[j] = nullptr;
  sa.a.master = in.master;
  sa.a.m = in.m;
  sa.a.v = in.v;
  sa.a.slot = in.slot;
  sa.a.lo = in.lo;
  sa.a.hi = in.hi;
  sa.a.world = in.world;
  sa.a.coef = in.coef;
  sa.a.skip = in.skip;
  sa.a.accum = in.accum;
  sa.a.invG = in.invG;
  sa.a.s = in.s;
  sa.a.win_lo = in.win.lo;
  sa.a.win_hi = in.win.hi;
  sa.t0 = (in.lo + T - 1) / T;
  sa.t1 = in.hi / T;
  sa.rag_lo[0] = in.lo;
  sa.rag_hi[0] = sa.t0 * T;
  sa.rag_lo[1] = sa.t1 * T;
  sa.rag_hi[1] = in.hi;
  sa.stages = stages;
  sa.stage_bytes = stage_bytes;
  sa.err = device_error_word();
  if (!sa.err) return cudaErrorInvalidSymbol;
  sa.a.err = sa.err;
  int64_t blocks = sa.t1 - sa.t0;
  if (blocks > (int64_t)sms * blocks_per_sm) blocks = (int64_t)sms * blocks_per_sm;
  return launch_kernel(kernel, dim3((unsigned)blocks), dim3(kStagedThreads), smem, stream, sa);
}

template <int GW, bool BF16G, int PD, int MAXN, bool ACC>
cudaError_t launch_one(const ShardStepLaunch& in, cudaStream_t stream) {
  // Resident blocks on the whole GPU for this instantiation, per device; the
  // grid is twice that, so the tail of one wave overlaps the next.
  static std::atomic<int> max_blocks_by_dev[64];
  auto kernel = shard_step_kernel<GW, BF16G, PD, MAXN, ACC>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int max_blocks = max_blocks_by_dev[dev & 63].load(std::memory_order_relaxed);
  if (max_blocks == 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
    if (e != cudaSuccess) return e;
    max_blocks = 2 * sms * (per_sm > 0 ? per_sm : 1);
    max_blocks_by_dev[dev & 63].store(max_blocks, std::memory_order_relaxed);
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
  a.win_lo = in.win.lo;
  a.win_hi = in.win.hi;
  a.err = ZS_BOUNDS_CHECK ? device_error_word() : nullptr;
  if (ZS_BOUNDS_CHECK && !a.err) return cudaErrorInvalidSymbol;
  const int64_t units = GW > 0 ? (in.hi - in.lo) / GW + 2 : (in.hi - in.lo);
  int64_t blocks = (units + kThreads - 1) / kThreads;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  return launch_kernel(kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, a);
}

// The staged path where it is eligible and (path 0) measured faster: N <= 50,
// 16-byte aligned state and slices, a slot aligned for its stores, two stages
// of some tile width that fit in shared memory (the widest is taken), at least
// 8 whole tiles of it.
template <bool BF16G, int PD, bool ACC>
bool try_staged(const ShardStepLaunch& a, cudaStream_t stream, cudaError_t* result) {
  const int path = step_path();
  if (path == 1 || a.world > kStagedMaxN) return false;
  uintptr_t ptrs = (uintptr_t)a.master | (uintptr_t)a.m | (uintptr_t)a.v | (uintptr_t)a.accum;
  for (int j = 0; j < a.world; ++j) ptrs |= (uintptr_t)a.grads[j];
  if (ptrs % 16 != 0) return false;
  // Per device: shared memory per SM (0 = not looked up yet), the opt-in
  // shared memory per block, the SM count.
  struct Shape {
    std::atomic<int> per_sm{0}, per_block{0}, sms{0};
  };
  static Shape shape_by_dev[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  Shape& sh = shape_by_dev[dev & 63];
  if (sh.per_sm.load(std::memory_order_acquire) == 0) {
    int per_sm = 0, per_block = 0, sms = 0;
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    sh.per_block.store(per_block, std::memory_order_relaxed);
    sh.sms.store(sms, std::memory_order_relaxed);
    sh.per_sm.store(per_sm, std::memory_order_release);
  }
  // The call's algorithmic bytes against twice the L2 (the launch shape).
  const int64_t call_bytes =
      (a.hi - a.lo) * ((int64_t)a.world * (BF16G ? 2 : 4) + (ACC ? 28 : 24) +
                       (PD == kParamBf16 ? 2 : PD == kParamFp32 ? 4 : 3));
  const bool small = call_bytes < (int64_t(256) << 20);
  // The widest tile (E = 4 or 2 elements per consumer thread) of which two
  // stages fit, with at least 8 whole tiles in the range and a slot aligned
  // for one thread's parameter stores. (4096-element tiles, E = 8, measured
  // slower on GB300: Llama-7B 0.926 against 1.042, GPT-2-small 0.835 against
  // 1.001 of the copy bandwidth.)
  int E = 0, stages = 0, per_sm_blocks = 0;
  uint32_t stage_bytes = 0;
  for (int e = 4; e >= 2 && E == 0; e /= 2) {
    const uint32_t t = (uint32_t)staged_tile(e);
    const uint32_t sb = (uint32_t)a.world * t * (BF16G ? 2u : 4u) + (ACC ? 4u : 3u) * t * 4u;
    int st = 0, bps = 0;
    staged_shape(sb, sh.per_sm.load(std::memory_order_relaxed),
                 sh.per_block.load(std::memory_order_relaxed), small, &st, &bps);
    if (st < 2 || a.hi / t - (a.lo + t - 1) / t < 8) continue;
    const uintptr_t slot_align = PD == kParamBf16 ? 2u * e : PD == kParamFp32 ? 4u * e : e;
    if ((uintptr_t)a.slot % slot_align != 0) continue;
    E = e;
    stages = st;
    per_sm_blocks = bps;
    stage_bytes = sb;
  }
  if (E == 0) return false;
  const int64_t T = staged_tile(E);
  // The per-call choice, from GB300 sweeps of both kernels (shard sizes 2^20 ..
  // 2^30 x N in 2..64 x slice and parameter dtypes, CUDA graphs of 20 steps)
  // and the named workloads' step, accumulated and clipped pipelines. The
  // staged kernel is faster nearly everywhere with
  // 2048-element tiles (2^24 elements, N = 8 bf16: 1.002 against 0.897 of the
  // copy bandwidth; the GPT-2-small step 1.00 against 0.87; Llama-7B 1.041
  // against 1.014); the register-streaming kernel keeps fp32 slices with N <= 4
  // from 2^25 elements (2^26, N = 4: 1.006 against 0.977; with fp32 parameters
  // 1.015 against 0.958) and fp32 parameters from bf16 slices with N = 4..8 from
  // 2^26 (2^30, N = 8: 1.026 against 1.011), where it is ahead by up to 1.5 %;
  // below 2^26 the staged kernel is ahead there too (2^24, N = 2 / 4 / 8: 0.913 /
  // 0.969 / 0.959 against 0.823 / 0.906 / 0.911). With 1024-element
  // tiles (more slices than two 2048-element stages hold) the staged kernel wins
  // under 2^25 elements with bf16 slices (N = 48 at 2^24: 1.018 against 0.970)
  // and loses above (N = 32 at 2^26: 0.997 against 1.017); with fp32 slices it
  // wins or ties.
  const int64_t len = a.hi - a.lo;
  const bool direct_wins =
      E == 4 ? (!BF16G && a.world <= 4 && len >= (int64_t(1) << 25)) ||
                   (BF16G && PD == kParamFp32 && a.world >= 4 && a.world <= 8 &&
                    len >= (int64_t(1) << 26))
             : BF16G && len >= (int64_t(1) << 25);
  if (path == 0 && direct_wins) return false;
  const int sms = sh.sms.load(std::memory_order_relaxed);
  const int smem_sm = sh.per_sm.load(std::memory_order_relaxed);
  if (E == 4)
    *result = launch_staged<BF16G, PD, ACC, 4>(a, stage_bytes, stages, per_sm_blocks, sms, smem_sm,
                                               stream);
  else
    *result = launch_staged<BF16G, PD, ACC, 2>(a, stage_bytes, stages, per_sm_blocks, sms, smem_sm,
                                               stream);
  if (*result == cudaSuccess) note_step_kernel(2, (int)T);
  return true;
}

template <bool BF16G, int PD, bool ACC>
cudaError_t dispatch(const ShardStepLaunch& a, cudaStream_t stream) {
  cudaError_t staged_result = cudaSuccess;
  if (try_staged<BF16G, PD, ACC>(a, stream, &staged_result)) return staged_result;
  cudaError_t e;
  // Slice-pointer tables sized to the world (the table is the launch's
  // parameter block: 128 B, 512 B or 8 KB).
  if (a.vec_width == 16)
    e = a.world <= 16   ? launch_one<16, BF16G, PD, 16, ACC>(a, stream)
        : a.world <= 64 ? launch_one<16, BF16G, PD, 64, ACC>(a, stream)
                        : launch_one<16, BF16G, PD, ZS_MAX_WORLD, ACC>(a, stream);
  else if (a.vec_width == 8)
    e = launch_one<8, BF16G, PD, ZS_MAX_WORLD, ACC>(a, stream);
  else
    e = launch_one<0, BF16G, PD, ZS_MAX_WORLD, ACC>(a, stream);
  if (e == cudaSuccess) note_step_kernel(1, a.vec_width);
  return e;
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
