// shard_step.cu — the fused shard-local step: N-slice fp32 mean + AdamW on the
// fp32 master/m/v shard + cast of the updated master into this rank's slot of
// the AllGather buffer, in one memory-bound pass.
//
// The step ("从 Data Parallel 到 ZeRO/FSDP", "ZeRO Stage 1": after the gradient
// ReduceScatter the owner rank updates its optimizer/parameter shard, then
// all-gathers the updated parameters; "ZeRO vs FSDP: A Rigorous Dissection",
// §2.1-2.3) touches each shard element once: it reads N incoming gradient
// values and the fp32 master, m and v, and writes master, m, v and one
// low-precision parameter: g*N + 24 + p bytes per element and about N + 15
// flops, so HBM bandwidth bounds it and no tensor-core work exists here.
//
// Layout of the work: the shard-local range [lo, hi) is cut into groups of 8
// elements (16 bytes of bf16 per slice). A persistent grid walks the groups
// with a grid stride; each group is one thread's 16-byte vector loads of every
// slice and of the three states, the fp32 arithmetic, and 16-byte vector
// stores. Elements before the first and after the last whole group (bucket
// ranges start and end at tensor boundaries) are done one by one.
//
// Arithmetic: every operation is an IEEE binary32 op rounded to nearest even
// (the _rn intrinsics are never contracted into FMAs), in the order the
// method fixes, so results are reproducible bit for bit.
#include <cuda_runtime.h>
#include <stdint.h>

#include "zs_internal.h"

namespace zs {

// Set by bounds-checked builds; read and cleared by zs_check_device_error.
__device__ unsigned int g_error_word;

namespace {

constexpr int kThreads = 256;
constexpr int kGroup = 8;   // elements per group
constexpr int kBatch = 8;   // gradient slices loaded back to back

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
  StepScalars s;
};

// ---- loads and stores ------------------------------------------------------
// Gradient slices are read-only for the kernel's lifetime and read once.
__device__ __forceinline__ uint4 ld_once(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
__device__ __forceinline__ float4 ld_state(const float* p) {
  float4 r;
  asm("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
      : "l"(p));
  return r;
}
__device__ __forceinline__ void st_state(float* p, float4 x) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(x.x), "f"(x.y),
               "f"(x.z), "f"(x.w)
               : "memory");
}
__device__ __forceinline__ void st_u32x4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                         uint32_t d) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void st_u32x2(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
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

// ---- one group of 8 elements -------------------------------------------------
// acc[k] += slice_j[8g + k] for j ascending. NG > 0: N known at compile time.
template <bool BF16G, int NG, int MAXN>
__device__ __forceinline__ void reduce_group(const StepArgs<MAXN>& a, int64_t g, float acc[8]) {
  constexpr int W = BF16G ? 1 : 2;  // 16-byte words per slice per group
  const int n = NG > 0 ? NG : a.world;
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
#pragma unroll(NG > 0 ? (NG + kBatch - 1) / kBatch : 1)
  for (int j0 = 0; j0 < n; j0 += kBatch) {
    uint4 raw[kBatch][W];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (j0 + b < n) {
        const unsigned char* base =
            static_cast<const unsigned char*>(a.grads[j0 + b]) + g * (16 * W);
#pragma unroll
        for (int w = 0; w < W; ++w) raw[b][w] = ld_once(base + 16 * w);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (j0 + b < n) {
        if (BF16G) {
          const uint32_t q[4] = {raw[b][0].x, raw[b][0].y, raw[b][0].z, raw[b][0].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[2 * k] = __fadd_rn(acc[2 * k], bf16_lo(q[k]));
            acc[2 * k + 1] = __fadd_rn(acc[2 * k + 1], bf16_hi(q[k]));
          }
        } else {
#pragma unroll
          for (int w = 0; w < W; ++w) {
            acc[4 * w + 0] = __fadd_rn(acc[4 * w + 0], __uint_as_float(raw[b][w].x));
            acc[4 * w + 1] = __fadd_rn(acc[4 * w + 1], __uint_as_float(raw[b][w].y));
            acc[4 * w + 2] = __fadd_rn(acc[4 * w + 2], __uint_as_float(raw[b][w].z));
            acc[4 * w + 3] = __fadd_rn(acc[4 * w + 3], __uint_as_float(raw[b][w].w));
          }
        }
      }
    }
  }
}

template <int PD>
__device__ __forceinline__ void store_params8(unsigned char* slot, int64_t g, const float p[8]) {
  if (PD == kParamBf16) {
    st_u32x4(slot + 16 * g, pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
             pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7]));
  } else if (PD == kParamFp32) {
    st_state(reinterpret_cast<float*>(slot) + 8 * g, make_float4(p[0], p[1], p[2], p[3]));
    st_state(reinterpret_cast<float*>(slot) + 8 * g + 4, make_float4(p[4], p[5], p[6], p[7]));
  } else {
    uint32_t q[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) q[k] = to_fp24(p[k]);
    unsigned char* d = slot + 24 * g;  // 8-byte aligned
    st_u32x2(d, q[0] | (q[1] << 24), (q[1] >> 8) | (q[2] << 16));
    st_u32x2(d + 8, (q[2] >> 16) | (q[3] << 8), q[4] | (q[5] << 24));
    st_u32x2(d + 16, (q[5] >> 8) | (q[6] << 16), (q[6] >> 16) | (q[7] << 8));
  }
}

template <bool BF16G, int PD, int NG, int MAXN>
__device__ __forceinline__ void process_group(const StepArgs<MAXN>& a, int64_t g) {
  const float4 p0 = ld_state(a.master + 8 * g), p1 = ld_state(a.master + 8 * g + 4);
  const float4 m0 = ld_state(a.m + 8 * g), m1 = ld_state(a.m + 8 * g + 4);
  const float4 v0 = ld_state(a.v + 8 * g), v1 = ld_state(a.v + 8 * g + 4);
  float acc[8];
  reduce_group<BF16G, NG>(a, g, acc);
  float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
  float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
  float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int k = 0; k < 8; ++k) adamw(a.s, __fmul_rn(acc[k], a.s.invN), p[k], m[k], v[k]);
  st_state(a.master + 8 * g, make_float4(p[0], p[1], p[2], p[3]));
  st_state(a.master + 8 * g + 4, make_float4(p[4], p[5], p[6], p[7]));
  st_state(a.m + 8 * g, make_float4(m[0], m[1], m[2], m[3]));
  st_state(a.m + 8 * g + 4, make_float4(m[4], m[5], m[6], m[7]));
  st_state(a.v + 8 * g, make_float4(v[0], v[1], v[2], v[3]));
  st_state(a.v + 8 * g + 4, make_float4(v[4], v[5], v[6], v[7]));
  store_params8<PD>(a.slot, g, p);
}

// One element, for the ragged head/tail and unaligned slots.
template <bool BF16G, int PD, int MAXN>
__device__ __forceinline__ void process_element(const StepArgs<MAXN>& a, int64_t i) {
  float acc = 0.0f;
  for (int j = 0; j < a.world; ++j) {
    const float x = BF16G ? __uint_as_float(
                                (uint32_t) static_cast<const uint16_t*>(a.grads[j])[i] << 16)
                          : static_cast<const float*>(a.grads[j])[i];
    acc = __fadd_rn(acc, x);
  }
  float p = a.master[i], m = a.m[i], v = a.v[i];
  adamw(a.s, __fmul_rn(acc, a.s.invN), p, m, v);
  a.master[i] = p;
  a.m[i] = m;
  a.v[i] = v;
  if (PD == kParamBf16) {
    reinterpret_cast<uint16_t*>(a.slot)[i] = to_bf16(p);
  } else if (PD == kParamFp32) {
    reinterpret_cast<float*>(a.slot)[i] = p;
  } else {
    const uint32_t q = to_fp24(p);
    unsigned char* d = a.slot + 3 * i;
    d[0] = (unsigned char)(q & 0xFFu);
    d[1] = (unsigned char)((q >> 8) & 0xFFu);
    d[2] = (unsigned char)((q >> 16) & 0xFFu);
  }
}

template <bool BF16G, int PD, int NG, int MAXN, bool VEC>
__global__ void __launch_bounds__(kThreads)
    shard_step_kernel(const __grid_constant__ StepArgs<MAXN> a) {
  const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  if (!VEC) {
    for (int64_t i = a.lo + tid; i < a.hi; i += stride) process_element<BF16G, PD>(a, i);
    return;
  }
  int64_t g0 = (a.lo + kGroup - 1) / kGroup, g1 = a.hi / kGroup;
  if (g0 >= g1) {  // no whole group: everything is ragged
    for (int64_t i = a.lo + tid; i < a.hi; i += stride) process_element<BF16G, PD>(a, i);
    return;
  }
  const int64_t head = g0 * kGroup - a.lo, tail = a.hi - g1 * kGroup;
  if (tid < head) process_element<BF16G, PD>(a, a.lo + tid);
  else if (tid < head + tail) process_element<BF16G, PD>(a, g1 * kGroup + (tid - head));
  for (int64_t g = g0 + tid; g < g1; g += stride) process_group<BF16G, PD, NG>(a, g);
}

template <bool BF16G, int PD, int NG, int MAXN, bool VEC>
cudaError_t launch_one(const ShardStepLaunch& in, cudaStream_t stream) {
  // Resident blocks on the whole GPU for this instantiation, per device.
  static int max_blocks_by_dev[64];
  auto kernel = shard_step_kernel<BF16G, PD, NG, MAXN, VEC>;
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
    max_blocks = sms * (per_sm > 0 ? per_sm : 1);
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
  a.s = in.s;
  const int64_t units = VEC ? (in.hi - in.lo) / kGroup + 2 : (in.hi - in.lo);
  int64_t blocks = (units + kThreads - 1) / kThreads;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <bool BF16G, int PD>
cudaError_t dispatch_n(const ShardStepLaunch& a, cudaStream_t stream) {
  if (!a.slot_vec_ok) return launch_one<BF16G, PD, 0, ZS_MAX_WORLD, false>(a, stream);
  if constexpr (BF16G && PD == kParamBf16) {
    if (a.world == 4) return launch_one<BF16G, PD, 4, 16, true>(a, stream);
    if (a.world == 8) return launch_one<BF16G, PD, 8, 16, true>(a, stream);
  }
  if (a.world <= 16) return launch_one<BF16G, PD, 0, 16, true>(a, stream);
  return launch_one<BF16G, PD, 0, ZS_MAX_WORLD, true>(a, stream);
}

}  // namespace

cudaError_t launch_shard_step(const ShardStepLaunch& a, cudaStream_t stream) {
  const bool bf16g = a.grad_dtype == ZS_BF16;
  switch (a.param_dtype) {
    case ZS_BF16:
      return bf16g ? dispatch_n<true, kParamBf16>(a, stream) : dispatch_n<false, kParamBf16>(a, stream);
    case ZS_FP32:
      return bf16g ? dispatch_n<true, kParamFp32>(a, stream) : dispatch_n<false, kParamFp32>(a, stream);
    case ZS_FP24:
      return bf16g ? dispatch_n<true, kParamFp24>(a, stream) : dispatch_n<false, kParamFp24>(a, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_device_error(cudaStream_t stream, unsigned int* word) {
  void* addr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&addr, g_error_word);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpy(word, addr, sizeof(unsigned int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(addr, 0, sizeof(unsigned int));
  return e;
}

}  // namespace zs
