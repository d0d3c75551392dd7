// api.cpp — the C ABI: argument validation, the per-step fp32 scalars, and
// dispatch to the kernels. Every check that can fail runs before any kernel is
// enqueued, so a bad call returns a status and leaves the GPU untouched.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "zs_internal.h"

namespace {

thread_local char g_err[512];
// Counts this thread's calls (clear_error opens a call): allocations checked
// once in a call are trusted for the rest of it.
thread_local uint64_t g_call = 0;
int32_t g_validation = 1;

typedef CUresult (*PFN_addressRange)(CUdeviceptr*, size_t*, CUdeviceptr);

PFN_addressRange address_range_fn() {
  static PFN_addressRange fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return (PFN_addressRange) nullptr;
    }
    return (PFN_addressRange)p;
  }();
  return fn;
}

struct Range {
  uintptr_t lo, hi;
  const char* name;
  int index;
  bool output;
};

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Device-resident, on the current device, and (where the driver can tell)
// [p, p+bytes) inside one allocation.
// Allocations already checked in this call (device memory on the current
// device, extent known): the N slices of a ReduceScatter output usually share
// one, so a call with many slices makes a few driver queries instead of 2N.
struct CheckedAllocation {
  uint64_t call;
  uintptr_t base, end;
};
thread_local CheckedAllocation g_checked[4];
thread_local int g_checked_next = 0;

zs_status check_device_buffer(const void* p, int64_t bytes, const char* fn, const char* name,
                              int index) {
  if (g_validation < 1 || bytes == 0) return ZS_OK;
  const uintptr_t lo = (uintptr_t)p, hi = lo + (uint64_t)bytes;
  for (const CheckedAllocation& c : g_checked)
    if (c.call == g_call && c.base <= lo && hi <= c.end) return ZS_OK;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return zs::fail(ZS_ERR_INVAL, "%s: %s[%d] is not a CUDA pointer", fn, name, index);
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return zs::fail(ZS_ERR_INVAL, "%s: %s[%d] is not device memory", fn, name, index);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return zs::fail(ZS_ERR_CUDA, "%s: cudaGetDevice failed", fn);
  }
  if (attr.type == cudaMemoryTypeDevice && attr.device != dev)
    return zs::fail(ZS_ERR_INVAL, "%s: %s[%d] lives on device %d, current device is %d", fn,
                    name, index, attr.device, dev);
  if (PFN_addressRange range = address_range_fn()) {
    CUdeviceptr base = 0;
    size_t size = 0;
    if (range(&base, &size, (CUdeviceptr)(uintptr_t)p) == CUDA_SUCCESS) {
      if ((uintptr_t)p + (uint64_t)bytes > (uintptr_t)base + size)
        return zs::fail(ZS_ERR_RANGE,
                        "%s: %s[%d] needs %lld bytes but its allocation ends %lld bytes after it",
                        fn, name, index, (long long)bytes,
                        (long long)((uintptr_t)base + size - (uintptr_t)p));
      g_checked[g_checked_next] = {g_call, (uintptr_t)base, (uintptr_t)base + size};
      g_checked_next = (g_checked_next + 1) % 4;
    }
  }
  return ZS_OK;
}

zs_status check_overlaps(const std::vector<Range>& rs, const char* fn) {
  for (size_t a = 0; a < rs.size(); ++a) {
    if (!rs[a].output || rs[a].lo == rs[a].hi) continue;
    for (size_t b = 0; b < rs.size(); ++b) {
      if (a == b || rs[b].lo == rs[b].hi) continue;
      if (rs[a].lo < rs[b].hi && rs[b].lo < rs[a].hi)
        return zs::fail(ZS_ERR_INVAL, "%s: %s[%d] overlaps %s[%d]", fn, rs[a].name,
                        rs[a].index, rs[b].name, rs[b].index);
    }
  }
  return ZS_OK;
}

// The plan, rank and shard-local range [lo, hi) of a call on a rank's shard.
zs_status check_call(const char* fn, const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi) {
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "%s: not a live plan", fn);
  if (rank < 0 || rank >= plan->world)
    return zs::fail(ZS_ERR_RANGE, "%s: rank %d not in [0, %d)", fn, rank, plan->world);
  if (lo < 0 || hi < lo || hi > plan->S)
    return zs::fail(ZS_ERR_RANGE, "%s: [lo, hi) = [%lld, %lld) not inside [0, %lld)", fn,
                    (long long)lo, (long long)hi, (long long)plan->S);
  return ZS_OK;
}

// The N incoming slices of S elements of gb bytes: non-NULL and 16-byte
// aligned; their byte ranges go to `ranges` for the overlap check, and
// *all32 is cleared unless every one is 32-byte aligned.
zs_status check_slices(const char* fn, int32_t N, int64_t S, const void* const* grad_slices,
                       int gb, std::vector<Range>* ranges, bool* all32) {
  for (int32_t j = 0; j < N; ++j) {
    const void* g = grad_slices[j];
    if (!g) return zs::fail(ZS_ERR_INVAL, "%s: grad_slices[%d] is NULL", fn, j);
    if (!aligned16(g))
      return zs::fail(ZS_ERR_ALIGN, "%s: grad_slices[%d] is not 16-byte aligned", fn, j);
    *all32 = *all32 && (uintptr_t)g % 32 == 0;
    ranges->push_back({(uintptr_t)g, (uintptr_t)g + (uint64_t)S * gb, "grad_slices", j, false});
  }
  return ZS_OK;
}

// After the overlap check: each slice is device memory covering its bytes.
zs_status check_slices_resident(const char* fn, int32_t N, int64_t S,
                                const void* const* grad_slices, int gb) {
  for (int32_t j = 0; j < N; ++j)
    if (zs_status st = check_device_buffer(grad_slices[j], S * gb, fn, "grad_slices", j))
      return st;
  return ZS_OK;
}

// beta^t by right-to-left binary powering in IEEE double.
double pow_binary(double base, int64_t e) {
  double r = 1.0;
  while (e > 0) {
    if (e & 1) r = r * base;
    base = base * base;
    e >>= 1;
  }
  return r;
}

}  // namespace

namespace zs {

zs_status check_device_array(const void* p, int64_t bytes, const char* fn, const char* name) {
  return check_device_buffer(p, bytes, fn, name, 0);
}

zs_status fail(zs_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() {
  g_err[0] = '\0';
  ++g_call;
}

int elem_bytes(zs_dtype dt) {
  switch (dt) {
    case ZS_BF16: return 2;
    case ZS_FP32: return 4;
    case ZS_FP24: return 3;
  }
  return 0;
}

}  // namespace zs

namespace {

zs_status shard_step_impl(const char* fn, const zs_plan* plan, int32_t rank, int64_t lo,
                          int64_t hi, const void* const* grad_slices, zs_dtype grad_dtype,
                          float* master, float* exp_avg, float* exp_avg_sq, void* full_flat,
                          zs_dtype param_dtype, const zs_adamw_hparams* hp, int64_t step,
                          const float* coef, const int32_t* skip, const float* accum,
                          int32_t micro_steps, void* cuda_stream, bool shard_only = false) {
  zs::clear_error();
  if (zs_status st = check_call(fn, plan, rank, lo, hi)) return st;
  const int32_t N = plan->world;
  const int64_t S = plan->S;
  if (step < 1) return zs::fail(ZS_ERR_RANGE, "%s: step %lld < 1", fn, (long long)step);
  if (grad_dtype != ZS_BF16 && grad_dtype != ZS_FP32)
    return zs::fail(ZS_ERR_INVAL, "%s: gradient dtype %d is not bf16 or fp32", fn, (int)grad_dtype);
  const int pb = zs::elem_bytes(param_dtype);
  if (!pb) return zs::fail(ZS_ERR_INVAL, "%s: unknown parameter dtype %d", fn, (int)param_dtype);
  if (!hp) return zs::fail(ZS_ERR_INVAL, "%s: hyper-parameters are NULL", fn);
  if (!std::isfinite(hp->lr) || !std::isfinite(hp->weight_decay) || !std::isfinite(hp->eps) ||
      hp->eps < 0 || !(hp->beta1 >= 0 && hp->beta1 < 1) || !(hp->beta2 >= 0 && hp->beta2 < 1))
    return zs::fail(ZS_ERR_INVAL,
                    "%s: need finite lr/wd, eps >= 0 and betas in [0, 1) "
                    "(lr %g, beta1 %g, beta2 %g, eps %g, wd %g)",
                    fn, hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay);
  if (lo == hi) return ZS_OK;
  if (!grad_slices || !master || !exp_avg || !exp_avg_sq || !full_flat)
    return zs::fail(ZS_ERR_INVAL, "%s: NULL buffer", fn);
  const int gb = grad_dtype == ZS_BF16 ? 2 : 4;
  std::vector<Range> ranges;
  ranges.reserve(N + 4);
  bool slices32 = true;
  if (zs_status st = check_slices(fn, N, S, grad_slices, gb, &ranges, &slices32)) return st;
  const void* outs[4] = {master, exp_avg, exp_avg_sq, full_flat};
  // full_flat: the flat buffer of all N slots, or (shard_only) the rank's own
  // parameter shard of S elements.
  const char* names[4] = {"master", "exp_avg", "exp_avg_sq",
                          shard_only ? "param_shard" : "full_flat"};
  const int64_t out_bytes[4] = {S * 4, S * 4, S * 4, (shard_only ? S : plan->P_pad) * pb};
  for (int k = 0; k < 4; ++k) {
    if (!aligned16(outs[k])) return zs::fail(ZS_ERR_ALIGN, "%s: %s is not 16-byte aligned", fn, names[k]);
    ranges.push_back({(uintptr_t)outs[k], (uintptr_t)outs[k] + (uint64_t)out_bytes[k], names[k], 0, true});
  }
  if (accum) {
    if (!aligned16(accum)) return zs::fail(ZS_ERR_ALIGN, "%s: accum is not 16-byte aligned", fn);
    ranges.push_back({(uintptr_t)accum, (uintptr_t)accum + (uint64_t)S * 4, "accum", 0, false});
  }
  if (zs_status st = check_overlaps(ranges, fn)) return st;
  if (zs_status st = check_slices_resident(fn, N, S, grad_slices, gb)) return st;
  for (int k = 0; k < 4; ++k)
    if (zs_status st = check_device_buffer(outs[k], out_bytes[k], fn, names[k], 0)) return st;
  if (accum)
    if (zs_status st = check_device_buffer(accum, S * 4, fn, "accum", 0)) return st;

  zs::ShardStepLaunch a;
  a.grads = grad_slices;
  a.world = N;
  a.grad_dtype = grad_dtype;
  a.param_dtype = param_dtype;
  a.master = master;
  a.m = exp_avg;
  a.v = exp_avg_sq;
  a.slot = static_cast<unsigned char*>(full_flat) + (shard_only ? 0 : (uint64_t)rank * S * pb);
  a.lo = lo;
  a.hi = hi;
  a.win = zs::step_window(lo, hi);
  // The widest vector path every pointer allows: 32-byte accesses need all
  // bases (and the slot's 16-element groups) 32-byte aligned; 16-byte
  // accesses need the slot's 8-element groups aligned; else element by element.
  const bool all32 = slices32 && ((uintptr_t)master | (uintptr_t)exp_avg |
                                   (uintptr_t)exp_avg_sq | (uintptr_t)accum) % 32 == 0;
  const uintptr_t slot_addr = (uintptr_t)a.slot;
  if (all32 && slot_addr % (pb == 3 ? 16u : 32u) == 0)
    a.vec_width = 16;
  else if (slot_addr % (pb == 3 ? 8u : 16u) == 0)
    a.vec_width = 8;
  else
    a.vec_width = 0;
  a.s.b1 = (float)hp->beta1;
  a.s.b2 = (float)hp->beta2;
  a.s.omb1 = (float)(1.0 - hp->beta1);
  a.s.omb2 = (float)(1.0 - hp->beta2);
  a.s.bc1 = (float)(1.0 - pow_binary(hp->beta1, step));
  a.s.bc2 = (float)(1.0 - pow_binary(hp->beta2, step));
  a.s.lr = (float)hp->lr;
  a.s.eps = (float)hp->eps;
  a.s.decay = (float)(1.0 - hp->lr * hp->weight_decay);
  a.s.invN = (float)(1.0 / (double)N);
  a.coef = coef;
  a.skip = skip;
  a.accum = accum;
  a.invG = (float)(1.0 / (double)(micro_steps > 0 ? micro_steps : 1));
  cudaError_t e = accum ? zs::launch_shard_step_accumulated(a, static_cast<cudaStream_t>(cuda_stream))
                        : zs::launch_shard_step(a, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess)
    return zs::fail(ZS_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ZS_OK;
}

// A device scalar the kernels read: aligned, device memory, in bounds.
zs_status check_device_scalar(const void* p, int64_t bytes, const char* fn, const char* name) {
  if (!p) return zs::fail(ZS_ERR_INVAL, "%s: %s is NULL", fn, name);
  if ((uintptr_t)p % (uintptr_t)bytes != 0)
    return zs::fail(ZS_ERR_ALIGN, "%s: %s is not %lld-byte aligned", fn, name, (long long)bytes);
  return check_device_buffer(p, bytes, fn, name, 0);
}

}  // namespace

static zs_status zs_shard_step_untraced(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                                   const void* const* grad_slices, zs_dtype grad_dtype,
                                   float* master, float* exp_avg, float* exp_avg_sq,
                                   void* full_flat, zs_dtype param_dtype,
                                   const zs_adamw_hparams* hp, int64_t step,
                                   void* cuda_stream) {
  return shard_step_impl("zs_shard_step", plan, rank, lo, hi, grad_slices, grad_dtype, master,
                         exp_avg, exp_avg_sq, full_flat, param_dtype, hp, step, nullptr, nullptr,
                         nullptr, 1, cuda_stream);
}

static zs_status zs_shard_step_to_shard_untraced(const zs_plan* plan, int32_t rank, int64_t lo,
                                            int64_t hi, const void* const* grad_slices,
                                            zs_dtype grad_dtype, float* master, float* exp_avg,
                                            float* exp_avg_sq, void* param_shard,
                                            zs_dtype param_dtype, const zs_adamw_hparams* hp,
                                            int64_t step, void* cuda_stream) {
  return shard_step_impl("zs_shard_step_to_shard", plan, rank, lo, hi, grad_slices, grad_dtype,
                         master, exp_avg, exp_avg_sq, param_shard, param_dtype, hp, step, nullptr,
                         nullptr, nullptr, 1, cuda_stream, true);
}

static zs_status zs_shard_step_clipped_untraced(const zs_plan* plan, int32_t rank, int64_t lo,
                                           int64_t hi, const void* const* grad_slices,
                                           zs_dtype grad_dtype, float* master, float* exp_avg,
                                           float* exp_avg_sq, void* full_flat,
                                           zs_dtype param_dtype, const zs_adamw_hparams* hp,
                                           int64_t step, const float* coef,
                                           const int32_t* skip, void* cuda_stream) {
  static const char* fn = "zs_shard_step_clipped";
  zs::clear_error();
  if (coef)
    if (zs_status st = check_device_scalar(coef, 4, fn, "coef")) return st;
  if (skip)
    if (zs_status st = check_device_scalar(skip, 4, fn, "skip")) return st;
  return shard_step_impl(fn, plan, rank, lo, hi, grad_slices, grad_dtype, master, exp_avg,
                         exp_avg_sq, full_flat, param_dtype, hp, step, coef, skip, nullptr, 1,
                         cuda_stream);
}

static zs_status zs_shard_step_accumulated_untraced(const zs_plan* plan, int32_t rank, int64_t lo,
                                               int64_t hi, const void* const* grad_slices,
                                               zs_dtype grad_dtype, const float* accum,
                                               int32_t micro_steps, float* master,
                                               float* exp_avg, float* exp_avg_sq,
                                               void* full_flat, zs_dtype param_dtype,
                                               const zs_adamw_hparams* hp, int64_t step,
                                               void* cuda_stream) {
  static const char* fn = "zs_shard_step_accumulated";
  zs::clear_error();
  if (micro_steps < 1)
    return zs::fail(ZS_ERR_RANGE, "%s: micro_steps %d < 1", fn, micro_steps);
  if (!accum && hi > lo) return zs::fail(ZS_ERR_INVAL, "%s: accum is NULL", fn);
  return shard_step_impl(fn, plan, rank, lo, hi, grad_slices, grad_dtype, master, exp_avg,
                         exp_avg_sq, full_flat, param_dtype, hp, step, nullptr, nullptr, accum,
                         micro_steps, cuda_stream);
}

static zs_status zs_grad_accumulate_untraced(const zs_plan* plan, int32_t rank, int64_t lo,
                                        int64_t hi, const void* const* grad_slices,
                                        zs_dtype grad_dtype, float* accum, int32_t first,
                                        void* cuda_stream) {
  static const char* fn = "zs_grad_accumulate";
  zs::clear_error();
  if (zs_status st = check_call(fn, plan, rank, lo, hi)) return st;
  const int32_t N = plan->world;
  const int64_t S = plan->S;
  if (grad_dtype != ZS_BF16 && grad_dtype != ZS_FP32)
    return zs::fail(ZS_ERR_INVAL, "%s: gradient dtype %d is not bf16 or fp32", fn, (int)grad_dtype);
  if (lo == hi) return ZS_OK;
  if (!grad_slices || !accum) return zs::fail(ZS_ERR_INVAL, "%s: NULL buffer", fn);
  if (!aligned16(accum)) return zs::fail(ZS_ERR_ALIGN, "%s: accum is not 16-byte aligned", fn);
  const int gb = grad_dtype == ZS_BF16 ? 2 : 4;
  std::vector<Range> ranges;
  bool all32 = (uintptr_t)accum % 32 == 0;
  if (zs_status st = check_slices(fn, N, S, grad_slices, gb, &ranges, &all32)) return st;
  ranges.push_back({(uintptr_t)accum, (uintptr_t)accum + (uint64_t)S * 4, "accum", 0, true});
  if (zs_status st = check_overlaps(ranges, fn)) return st;
  if (zs_status st = check_slices_resident(fn, N, S, grad_slices, gb)) return st;
  if (zs_status st = check_device_buffer(accum, S * 4, fn, "accum", 0)) return st;
  zs::ShardStepLaunch a = {};
  a.grads = grad_slices;
  a.world = N;
  a.grad_dtype = grad_dtype;
  a.param_dtype = ZS_BF16;
  a.lo = lo;
  a.hi = hi;
  a.win = zs::step_window(lo, hi);
  a.vec_width = all32 ? 16 : 8;
  a.accum = accum;
  a.invG = 1.0f;
  a.s.invN = (float)(1.0 / (double)N);
  cudaError_t e = zs::launch_grad_accumulate(a, first ? 1 : 0,
                                             static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess)
    return zs::fail(ZS_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ZS_OK;
}

extern "C" int64_t zs_grad_norm_workspace_bytes(void) { return zs::kNormWorkspaceBytes; }

namespace {
// The norm pass. Scratch: the caller's workspace, or (noalloc) the library's
// static device array. accum (with micro_steps) selects the norm of the
// accumulated step's gradient.
zs_status sqnorm_impl(const char* fn, const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                      const void* const* grad_slices, zs_dtype grad_dtype, const float* accum,
                      int32_t micro_steps, bool noalloc, void* workspace,
                      int64_t workspace_bytes, double* sqnorm_out, void* cuda_stream) {
  zs::clear_error();
  if (zs_status st = check_call(fn, plan, rank, lo, hi)) return st;
  const int32_t N = plan->world;
  const int64_t S = plan->S;
  if (grad_dtype != ZS_BF16 && grad_dtype != ZS_FP32)
    return zs::fail(ZS_ERR_INVAL, "%s: gradient dtype %d is not bf16 or fp32", fn, (int)grad_dtype);
  // The scratch one norm pass needs does not depend on the input's size, and
  // the library's static array holds it.
  static_assert(zs::kNormWorkspaceBytes <= zs::kNoAllocScratchBytes,
                "the no-alloc norm pass's scratch must fit its static array");
  if (!noalloc) {
    if (!workspace || workspace_bytes < zs::kNormWorkspaceBytes)
      return zs::fail(ZS_ERR_RANGE, "%s: workspace must hold %lld bytes", fn,
                      (long long)zs::kNormWorkspaceBytes);
    if (!aligned16(workspace))
      return zs::fail(ZS_ERR_ALIGN, "%s: workspace is not 16-byte aligned", fn);
  }
  if (zs_status st = check_device_scalar(sqnorm_out, 8, fn, "sqnorm_out")) return st;
  if (hi > lo && !grad_slices) return zs::fail(ZS_ERR_INVAL, "%s: grad_slices is NULL", fn);
  const int gb = grad_dtype == ZS_BF16 ? 2 : 4;
  std::vector<Range> ranges;
  bool all32 = true;
  if (hi > lo)
    if (zs_status st = check_slices(fn, N, S, grad_slices, gb, &ranges, &all32)) return st;
  if (accum && hi > lo) {
    if (!aligned16(accum)) return zs::fail(ZS_ERR_ALIGN, "%s: accum is not 16-byte aligned", fn);
    all32 = all32 && (uintptr_t)accum % 32 == 0;
    ranges.push_back({(uintptr_t)accum, (uintptr_t)accum + (uint64_t)S * 4, "accum", 0, false});
  }
  if (!noalloc)
    ranges.push_back({(uintptr_t)workspace,
                      (uintptr_t)workspace + (uint64_t)zs::kNormWorkspaceBytes, "workspace", 0,
                      true});
  ranges.push_back({(uintptr_t)sqnorm_out, (uintptr_t)sqnorm_out + 8, "sqnorm_out", 0, true});
  if (zs_status st = check_overlaps(ranges, fn)) return st;
  if (!noalloc)
    if (zs_status st = check_device_buffer(workspace, zs::kNormWorkspaceBytes, fn, "workspace", 0))
      return st;
  if (hi > lo)
    if (zs_status st = check_slices_resident(fn, N, S, grad_slices, gb)) return st;
  if (accum && hi > lo)
    if (zs_status st = check_device_buffer(accum, S * 4, fn, "accum", 0)) return st;
  zs::NormLaunch a = {};
  a.grads = grad_slices;
  a.world = N;
  a.grad_dtype = grad_dtype;
  a.lo = lo;
  a.hi = hi;
  a.win = zs::step_window(lo, hi);
  a.vec = all32;
  a.invN = (float)(1.0 / (double)N);
  a.accum = hi > lo ? accum : nullptr;
  a.invG = (float)(1.0 / (double)(micro_steps > 0 ? micro_steps : 1));
  a.out = sqnorm_out;
  cudaError_t e;
  if (noalloc) {
    // partials and ticket: set to the static array by the launcher
    e = zs::launch_grad_sqnorm_noalloc(a, static_cast<cudaStream_t>(cuda_stream));
  } else {
    a.partials = static_cast<double*>(workspace);
    a.ticket = reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(workspace) +
                                               zs::kNormTicketOffset);
    e = zs::launch_grad_sqnorm(a, static_cast<cudaStream_t>(cuda_stream));
  }
  if (e != cudaSuccess)
    return zs::fail(ZS_ERR_CUDA, "%s: %s failed: %s", fn, noalloc ? "set-up or launch" : "launch",
                    cudaGetErrorString(e));
  return ZS_OK;
}
}  // namespace

static zs_status zs_grad_sqnorm_untraced(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                                         const void* const* grad_slices, zs_dtype grad_dtype,
                                         void* workspace, int64_t workspace_bytes,
                                         double* sqnorm_out, void* cuda_stream) {
  return sqnorm_impl("zs_grad_sqnorm", plan, rank, lo, hi, grad_slices, grad_dtype, nullptr, 1,
                     false, workspace, workspace_bytes, sqnorm_out, cuda_stream);
}

static zs_status zs_grad_sqnorm_accumulated_untraced(
    const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi, const void* const* grad_slices,
    zs_dtype grad_dtype, const float* accum, int32_t micro_steps, void* workspace,
    int64_t workspace_bytes, double* sqnorm_out, void* cuda_stream) {
  static const char* fn = "zs_grad_sqnorm_accumulated";
  zs::clear_error();
  if (micro_steps < 1) return zs::fail(ZS_ERR_RANGE, "%s: micro_steps %d < 1", fn, micro_steps);
  if (!accum && hi > lo) return zs::fail(ZS_ERR_INVAL, "%s: accum is NULL", fn);
  return sqnorm_impl(fn, plan, rank, lo, hi, grad_slices, grad_dtype, accum, micro_steps, false,
                     workspace, workspace_bytes, sqnorm_out, cuda_stream);
}

static zs_status zs_shard_step_accumulated_clipped_untraced(
    const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi, const void* const* grad_slices,
    zs_dtype grad_dtype, const float* accum, int32_t micro_steps, float* master, float* exp_avg,
    float* exp_avg_sq, void* full_flat, zs_dtype param_dtype, const zs_adamw_hparams* hp,
    int64_t step, const float* coef, const int32_t* skip, void* cuda_stream) {
  static const char* fn = "zs_shard_step_accumulated_clipped";
  zs::clear_error();
  if (micro_steps < 1) return zs::fail(ZS_ERR_RANGE, "%s: micro_steps %d < 1", fn, micro_steps);
  if (!accum && hi > lo) return zs::fail(ZS_ERR_INVAL, "%s: accum is NULL", fn);
  if (coef)
    if (zs_status st = check_device_scalar(coef, 4, fn, "coef")) return st;
  if (skip)
    if (zs_status st = check_device_scalar(skip, 4, fn, "skip")) return st;
  return shard_step_impl(fn, plan, rank, lo, hi, grad_slices, grad_dtype, master, exp_avg,
                         exp_avg_sq, full_flat, param_dtype, hp, step, coef, skip, accum,
                         micro_steps, cuda_stream);
}

static zs_status zs_grad_sqnorm_noalloc_untraced(const zs_plan* plan, int32_t rank, int64_t lo,
                                                 int64_t hi, const void* const* grad_slices,
                                                 zs_dtype grad_dtype, double* sqnorm_out,
                                                 void* cuda_stream) {
  return sqnorm_impl("zs_grad_sqnorm_noalloc", plan, rank, lo, hi, grad_slices, grad_dtype,
                     nullptr, 1, true, nullptr, 0, sqnorm_out, cuda_stream);
}

static zs_status zs_clip_coefficient_untraced(const double* rank_sqnorms, int32_t n, double max_norm,
                                         float* coef_out, int32_t* nonfinite_out,
                                         void* cuda_stream) {
  static const char* fn = "zs_clip_coefficient";
  zs::clear_error();
  if (n < 1 || n > ZS_MAX_WORLD) return zs::fail(ZS_ERR_RANGE, "%s: n %d outside 1..%d", fn, n, ZS_MAX_WORLD);
  if (!std::isfinite(max_norm) || !(max_norm > 0))
    return zs::fail(ZS_ERR_INVAL, "%s: max_norm must be finite and > 0 (got %g)", fn, max_norm);
  if (!rank_sqnorms || (uintptr_t)rank_sqnorms % 8)
    return zs::fail(ZS_ERR_ALIGN, "%s: rank_sqnorms must be 8-byte aligned device memory", fn);
  if (zs_status st = check_device_buffer(rank_sqnorms, 8 * (int64_t)n, fn, "rank_sqnorms", 0)) return st;
  if (zs_status st = check_device_scalar(coef_out, 4, fn, "coef_out")) return st;
  if (zs_status st = check_device_scalar(nonfinite_out, 4, fn, "nonfinite_out")) return st;
  cudaError_t e = zs::launch_clip_coef(rank_sqnorms, n, max_norm, coef_out, nonfinite_out,
                                       static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess)
    return zs::fail(ZS_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ZS_OK;
}

static zs_status zs_gather_assemble_untraced(const zs_plan* plan, int32_t rank,
                                        const void* const* shard_srcs, void* full_flat,
                                        zs_dtype param_dtype, void** views_out,
                                        void* cuda_stream) {
  static const char* fn = "zs_gather_assemble";
  zs::clear_error();
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "%s: not a live plan", fn);
  const int32_t N = plan->world;
  if (rank < 0 || rank >= N) return zs::fail(ZS_ERR_RANGE, "%s: rank %d not in [0, %d)", fn, rank, N);
  const int pb = zs::elem_bytes(param_dtype);
  if (!pb) return zs::fail(ZS_ERR_INVAL, "%s: unknown parameter dtype %d", fn, (int)param_dtype);
  if (!full_flat) return zs::fail(ZS_ERR_INVAL, "%s: full_flat is NULL", fn);
  if (!aligned16(full_flat)) return zs::fail(ZS_ERR_ALIGN, "%s: full_flat is not 16-byte aligned", fn);
  if (!shard_srcs && N > 1) return zs::fail(ZS_ERR_INVAL, "%s: shard_srcs is NULL", fn);
  const int64_t slot_bytes = plan->S * pb;
  unsigned char* dst = static_cast<unsigned char*>(full_flat);
  const uintptr_t dlo = (uintptr_t)dst, dhi = dlo + (uint64_t)plan->P_pad * pb;
  std::vector<const unsigned char*> srcs(N, nullptr);
  int active = 0;
  if (slot_bytes > 0) {
    if (zs_status st = check_device_buffer(full_flat, plan->P_pad * pb, fn, "full_flat", 0)) return st;
    for (int32_t j = 0; j < N; ++j) {
      const unsigned char* s = shard_srcs ? static_cast<const unsigned char*>(shard_srcs[j]) : nullptr;
      if (j == rank || !s || s == dst + (uint64_t)j * slot_bytes) continue;
      if (!aligned16(s)) return zs::fail(ZS_ERR_ALIGN, "%s: shard_srcs[%d] is not 16-byte aligned", fn, j);
      const uintptr_t slo = (uintptr_t)s, shi = slo + (uint64_t)slot_bytes;
      if (slo < dhi && dlo < shi)
        return zs::fail(ZS_ERR_INVAL, "%s: shard_srcs[%d] overlaps full_flat", fn, j);
      if (zs_status st = check_device_buffer(s, slot_bytes, fn, "shard_srcs", j)) return st;
      srcs[j] = s;
      ++active;
    }
  }
  if (active > 0) {
    zs::GatherLaunch g;
    g.srcs = srcs.data();
    g.world = N;
    g.dst = dst;
    g.slot_bytes = slot_bytes;
    cudaError_t e = zs::launch_gather(g, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess)
      return zs::fail(ZS_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  }
  if (views_out) {
    if (plan->layout != zs::kLayoutFlat)
      return zs::fail(ZS_ERR_UNSUPPORTED,
                      "%s: a row-sharded plan's gathered buffer is rank-major; zs_unshard copies "
                      "it out into parameters (views_out must be NULL)", fn);
    for (int32_t k = 0; k < plan->n_params; ++k)
      views_out[k] = dst + (uint64_t)plan->offsets[k] * pb;
  }
  return ZS_OK;
}

namespace {

// Rows [r*c, min((r+1)*c, d)) of a parameter with d rows of w elements.
int64_t valid_rows(const zs_plan* p, int32_t i, int32_t r) {
  const int64_t c = p->rows_per_rank[i], d = p->dim0[i];
  const int64_t lo = (int64_t)r * c;
  if (lo >= d) return 0;
  return (lo + c <= d ? c : d - lo);
}

zs_status check_rows_params(const zs_plan* plan, const void* const* params, int pb, bool output,
                            const char* fn, std::vector<Range>* ranges) {
  if (!params && plan->n_params > 0) return zs::fail(ZS_ERR_INVAL, "%s: parameter list is NULL", fn);
  for (int32_t i = 0; i < plan->n_params; ++i) {
    if (plan->owner[i] != i || plan->numels[i] == 0) continue;
    const void* q = params[i];
    if (!q) return zs::fail(ZS_ERR_INVAL, "%s: params[%d] is NULL", fn, i);
    const uintptr_t need = pb == 3 ? 1u : (uintptr_t)pb;  // 3-byte elements: any byte
    if ((uintptr_t)q % need)
      return zs::fail(ZS_ERR_ALIGN, "%s: params[%d] is not %d-byte aligned", fn, i, (int)need);
    const int64_t bytes = plan->numels[i] * pb;
    ranges->push_back({(uintptr_t)q, (uintptr_t)q + (uint64_t)bytes, "params", i, output});
    if (zs_status st = check_device_buffer(q, bytes, fn, "params", i)) return st;
  }
  return ZS_OK;
}

}  // namespace

static zs_status zs_unshard_untraced(const zs_plan* plan, const void* gathered, zs_dtype dtype,
                                void* const* params_out, void* cuda_stream) {
  static const char* fn = "zs_unshard";
  zs::clear_error();
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "%s: not a live plan", fn);
  if (plan->layout != zs::kLayoutRows)
    return zs::fail(ZS_ERR_UNSUPPORTED, "%s: a flat plan's gathered buffer already is the "
                    "parameters (use the views of zs_gather_assemble)", fn);
  const int pb = zs::elem_bytes(dtype);
  if (!pb) return zs::fail(ZS_ERR_INVAL, "%s: unknown dtype %d", fn, (int)dtype);
  const int32_t N = plan->world;
  const int64_t S = plan->S;
  if (!gathered && S > 0) return zs::fail(ZS_ERR_INVAL, "%s: gathered is NULL", fn);
  if ((uintptr_t)gathered % 16) return zs::fail(ZS_ERR_ALIGN, "%s: gathered is not 16-byte aligned", fn);
  std::vector<Range> ranges;
  const int64_t gbytes = (int64_t)N * S * pb;
  ranges.push_back({(uintptr_t)gathered, (uintptr_t)gathered + (uint64_t)gbytes, "gathered", 0, false});
  if (zs_status st = check_rows_params(plan, (const void* const*)params_out, pb, true, fn, &ranges)) return st;
  if (zs_status st = check_overlaps(ranges, fn)) return st;
  if (zs_status st = check_device_buffer(gathered, gbytes, fn, "gathered", 0)) return st;
  std::vector<zs::RowSegment> segs;
  const unsigned char* g = static_cast<const unsigned char*>(gathered);
  for (int32_t i = 0; i < plan->n_params; ++i) {
    if (plan->owner[i] != i) continue;
    const int64_t w = plan->row_elems[i], c = plan->rows_per_rank[i];
    for (int32_t r = 0; r < N; ++r) {
      const int64_t rows = valid_rows(plan, i, r);
      if (rows == 0) continue;
      zs::RowSegment sg;
      sg.src = g + ((uint64_t)r * S + plan->offsets[i]) * pb;
      sg.dst = static_cast<unsigned char*>(params_out[i]) + (uint64_t)r * c * w * pb;
      sg.copy_bytes = rows * w * pb;
      sg.zero_bytes = 0;
      segs.push_back(sg);
    }
  }
  if (segs.empty()) return ZS_OK;
  cudaError_t e = zs::launch_segment_copy(segs.data(), (int)segs.size(),
                                          static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess)
    return zs::fail(ZS_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ZS_OK;
}

static zs_status zs_shard_rows_untraced(const zs_plan* plan, int32_t rank, const void* const* params_in,
                                   zs_dtype dtype, void* local_out, void* cuda_stream) {
  static const char* fn = "zs_shard_rows";
  zs::clear_error();
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "%s: not a live plan", fn);
  if (plan->layout != zs::kLayoutRows)
    return zs::fail(ZS_ERR_UNSUPPORTED, "%s: not a row-sharded plan", fn);
  const int pb = zs::elem_bytes(dtype);
  if (!pb) return zs::fail(ZS_ERR_INVAL, "%s: unknown dtype %d", fn, (int)dtype);
  const int32_t N = plan->world;
  const int64_t S = plan->S;
  if (rank < 0 || rank >= N) return zs::fail(ZS_ERR_RANGE, "%s: rank %d not in [0, %d)", fn, rank, N);
  if (S == 0) return ZS_OK;
  if (!local_out) return zs::fail(ZS_ERR_INVAL, "%s: local_out is NULL", fn);
  if ((uintptr_t)local_out % 16) return zs::fail(ZS_ERR_ALIGN, "%s: local_out is not 16-byte aligned", fn);
  std::vector<Range> ranges;
  ranges.push_back({(uintptr_t)local_out, (uintptr_t)local_out + (uint64_t)S * pb, "local_out", 0, true});
  if (zs_status st = check_rows_params(plan, params_in, pb, false, fn, &ranges)) return st;
  if (zs_status st = check_overlaps(ranges, fn)) return st;
  if (zs_status st = check_device_buffer(local_out, S * pb, fn, "local_out", 0)) return st;
  std::vector<zs::RowSegment> segs;
  unsigned char* out = static_cast<unsigned char*>(local_out);
  int64_t used = 0;
  for (int32_t i = 0; i < plan->n_params; ++i) {
    if (plan->owner[i] != i) continue;
    const int64_t w = plan->row_elems[i], c = plan->rows_per_rank[i];
    const int64_t rows = valid_rows(plan, i, rank);
    zs::RowSegment sg;
    sg.src = rows ? static_cast<const unsigned char*>(params_in[i]) + (uint64_t)rank * c * w * pb
                  : nullptr;
    sg.dst = out + (uint64_t)plan->offsets[i] * pb;
    sg.copy_bytes = rows * w * pb;
    sg.zero_bytes = (c - rows) * w * pb;
    used = plan->offsets[i] + c * w;
    if (sg.copy_bytes + sg.zero_bytes > 0) segs.push_back(sg);
  }
  if (S > used) {
    zs::RowSegment pad;
    pad.src = nullptr;
    pad.dst = out + (uint64_t)used * pb;
    pad.copy_bytes = 0;
    pad.zero_bytes = (S - used) * pb;
    segs.push_back(pad);
  }
  if (segs.empty()) return ZS_OK;
  cudaError_t e = zs::launch_segment_copy(segs.data(), (int)segs.size(),
                                          static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess)
    return zs::fail(ZS_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ZS_OK;
}

extern "C" const char* zs_status_string(zs_status st) {
  switch (st) {
    case ZS_OK: return "ok";
    case ZS_ERR_INVAL: return "invalid argument";
    case ZS_ERR_ALIGN: return "misaligned device pointer";
    case ZS_ERR_RANGE: return "out of range";
    case ZS_ERR_CUDA: return "CUDA error";
    case ZS_ERR_NOMEM: return "out of host memory";
    case ZS_ERR_TIMEOUT: return "device wait timed out";
    case ZS_ERR_UNSUPPORTED: return "unsupported";
    case ZS_ERR_IO: return "file I/O failed";
    case ZS_ERR_CORRUPT: return "checkpoint corrupt or inconsistent";
  }
  return "unknown status";
}

extern "C" const char* zs_last_error(void) { return g_err; }

extern "C" zs_status zs_check_device_error(void* cuda_stream) {
  zs::clear_error();
  unsigned int word = 0;
  cudaError_t e = zs::read_and_clear_device_error(static_cast<cudaStream_t>(cuda_stream), &word);
  if (e != cudaSuccess)
    return zs::fail(ZS_ERR_CUDA, "zs_check_device_error: %s", cudaGetErrorString(e));
  if (word & 2u) return zs::fail(ZS_ERR_TIMEOUT, "zs_check_device_error: a device wait timed out");
  if (word & 1u) return zs::fail(ZS_ERR_RANGE, "zs_check_device_error: a bounds check failed");
  return ZS_OK;
}

namespace {
std::atomic<int32_t> g_step_path{0};
std::atomic<int64_t> g_bounds_shrink{0};
}  // namespace

namespace zs {
int step_path() { return g_step_path.load(std::memory_order_relaxed); }

Window step_window(int64_t lo, int64_t hi) {
  const int64_t k = g_bounds_shrink.load(std::memory_order_relaxed);
  return Window{lo + k, hi - k};
}
}  // namespace zs

extern "C" int32_t zs_bounds_checked(void) { return zs::bounds_checked(); }

extern "C" zs_status zs_selftest_bounds_window(int64_t shrink) {
  zs::clear_error();
  if (!zs::bounds_checked())
    return zs::fail(ZS_ERR_UNSUPPORTED,
                    "zs_selftest_bounds_window: this library is not the bounds-checked build");
  if (shrink < 0 || shrink > (int64_t(1) << 40))
    return zs::fail(ZS_ERR_RANGE, "zs_selftest_bounds_window: shrink %lld outside 0..2^40",
                    (long long)shrink);
  g_bounds_shrink.store(shrink);
  return ZS_OK;
}

extern "C" zs_status zs_selftest_wait_timeout(uint32_t polls, void* cuda_stream) {
  zs::clear_error();
  if (polls == 0 || polls > (1u << 20))
    return zs::fail(ZS_ERR_RANGE, "zs_selftest_wait_timeout: polls %u outside 1..2^20", polls);
  const cudaError_t e = zs::launch_wait_timeout(polls, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess)
    return zs::fail(ZS_ERR_CUDA, "zs_selftest_wait_timeout: %s", cudaGetErrorString(e));
  return ZS_OK;
}

extern "C" int32_t zs_set_step_path(int32_t path) {
  if (path < 0 || path > 2) return -1;
  return g_step_path.exchange(path);
}

namespace {
thread_local int32_t t_last_kernel = 0, t_last_elems = 0;
std::atomic<int32_t> g_launch_overlap{1};
}  // namespace

namespace zs {
bool launch_overlap() { return g_launch_overlap.load(std::memory_order_relaxed) != 0; }
}  // namespace zs

extern "C" int32_t zs_set_launch_overlap(int32_t on) {
  if (on != 0 && on != 1) return -1;
  return g_launch_overlap.exchange(on);
}

namespace zs {
void note_step_kernel(int kernel, int elems) {
  t_last_kernel = kernel;
  t_last_elems = elems;
}
}  // namespace zs

extern "C" zs_status zs_last_step_kernel(int32_t* kernel, int32_t* elems) {
  zs::clear_error();
  if (!kernel || !elems) return zs::fail(ZS_ERR_INVAL, "zs_last_step_kernel: NULL output");
  *kernel = t_last_kernel;
  *elems = t_last_elems;
  return ZS_OK;
}

extern "C" int32_t zs_set_validation(int32_t level) {
  int32_t old = g_validation;
  g_validation = level;
  return old;
}

extern "C" const char* zs_version(void) { return "0.1.0"; }

// ---- traced entry points ----------------------------------------------------------
// Each call at a collective site of the real system leaves one record in the
// per-call trace (trace.cpp) with its status, whatever path it returned by.
extern "C" zs_status zs_shard_step(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                                   const void* const* grad_slices, zs_dtype grad_dtype,
                                   float* master, float* exp_avg, float* exp_avg_sq,
                                   void* full_flat, zs_dtype param_dtype,
                                   const zs_adamw_hparams* hp, int64_t step,
                                   void* cuda_stream) {
  const zs::CallRange range("zs_shard_step");
  return zs::traced(zs_shard_step_untraced(plan, rank, lo, hi, grad_slices, grad_dtype, master,
                                           exp_avg, exp_avg_sq, full_flat, param_dtype, hp,
                                           step, cuda_stream),
                    "zs_shard_step", plan, rank, lo, hi, grad_dtype, param_dtype, step);
}

extern "C" zs_status zs_shard_step_to_shard(const zs_plan* plan, int32_t rank, int64_t lo,
                                            int64_t hi, const void* const* grad_slices,
                                            zs_dtype grad_dtype, float* master, float* exp_avg,
                                            float* exp_avg_sq, void* param_shard,
                                            zs_dtype param_dtype, const zs_adamw_hparams* hp,
                                            int64_t step, void* cuda_stream) {
  const zs::CallRange range("zs_shard_step_to_shard");
  return zs::traced(zs_shard_step_to_shard_untraced(plan, rank, lo, hi, grad_slices, grad_dtype,
                                                    master, exp_avg, exp_avg_sq, param_shard,
                                                    param_dtype, hp, step, cuda_stream),
                    "zs_shard_step_to_shard", plan, rank, lo, hi, grad_dtype, param_dtype, step);
}

extern "C" zs_status zs_shard_step_clipped(const zs_plan* plan, int32_t rank, int64_t lo,
                                           int64_t hi, const void* const* grad_slices,
                                           zs_dtype grad_dtype, float* master, float* exp_avg,
                                           float* exp_avg_sq, void* full_flat,
                                           zs_dtype param_dtype, const zs_adamw_hparams* hp,
                                           int64_t step, const float* coef,
                                           const int32_t* skip, void* cuda_stream) {
  const zs::CallRange range("zs_shard_step_clipped");
  return zs::traced(zs_shard_step_clipped_untraced(plan, rank, lo, hi, grad_slices, grad_dtype,
                                                   master, exp_avg, exp_avg_sq, full_flat,
                                                   param_dtype, hp, step, coef, skip,
                                                   cuda_stream),
                    "zs_shard_step_clipped", plan, rank, lo, hi, grad_dtype, param_dtype, step);
}

extern "C" zs_status zs_shard_step_accumulated(const zs_plan* plan, int32_t rank, int64_t lo,
                                               int64_t hi, const void* const* grad_slices,
                                               zs_dtype grad_dtype, const float* accum,
                                               int32_t micro_steps, float* master,
                                               float* exp_avg, float* exp_avg_sq,
                                               void* full_flat, zs_dtype param_dtype,
                                               const zs_adamw_hparams* hp, int64_t step,
                                               void* cuda_stream) {
  const zs::CallRange range("zs_shard_step_accumulated");
  return zs::traced(zs_shard_step_accumulated_untraced(plan, rank, lo, hi, grad_slices,
                                                       grad_dtype, accum, micro_steps, master,
                                                       exp_avg, exp_avg_sq, full_flat,
                                                       param_dtype, hp, step, cuda_stream),
                    "zs_shard_step_accumulated", plan, rank, lo, hi, grad_dtype, param_dtype,
                    step);
}

extern "C" zs_status zs_grad_accumulate(const zs_plan* plan, int32_t rank, int64_t lo,
                                        int64_t hi, const void* const* grad_slices,
                                        zs_dtype grad_dtype, float* accum, int32_t first,
                                        void* cuda_stream) {
  const zs::CallRange range("zs_grad_accumulate");
  return zs::traced(zs_grad_accumulate_untraced(plan, rank, lo, hi, grad_slices, grad_dtype,
                                                accum, first, cuda_stream),
                    "zs_grad_accumulate", plan, rank, lo, hi, grad_dtype, -1, 0);
}

extern "C" zs_status zs_grad_sqnorm(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                                    const void* const* grad_slices, zs_dtype grad_dtype,
                                    void* workspace, int64_t workspace_bytes,
                                    double* sqnorm_out, void* cuda_stream) {
  const zs::CallRange range("zs_grad_sqnorm");
  return zs::traced(zs_grad_sqnorm_untraced(plan, rank, lo, hi, grad_slices, grad_dtype,
                                            workspace, workspace_bytes, sqnorm_out,
                                            cuda_stream),
                    "zs_grad_sqnorm", plan, rank, lo, hi, grad_dtype, -1, 0);
}

extern "C" zs_status zs_grad_sqnorm_accumulated(const zs_plan* plan, int32_t rank, int64_t lo,
                                                int64_t hi, const void* const* grad_slices,
                                                zs_dtype grad_dtype, const float* accum,
                                                int32_t micro_steps, void* workspace,
                                                int64_t workspace_bytes, double* sqnorm_out,
                                                void* cuda_stream) {
  const zs::CallRange range("zs_grad_sqnorm_accumulated");
  return zs::traced(zs_grad_sqnorm_accumulated_untraced(plan, rank, lo, hi, grad_slices,
                                                        grad_dtype, accum, micro_steps,
                                                        workspace, workspace_bytes, sqnorm_out,
                                                        cuda_stream),
                    "zs_grad_sqnorm_accumulated", plan, rank, lo, hi, grad_dtype, -1, 0);
}

extern "C" zs_status zs_shard_step_accumulated_clipped(
    const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi, const void* const* grad_slices,
    zs_dtype grad_dtype, const float* accum, int32_t micro_steps, float* master, float* exp_avg,
    float* exp_avg_sq, void* full_flat, zs_dtype param_dtype, const zs_adamw_hparams* hp,
    int64_t step, const float* coef, const int32_t* skip, void* cuda_stream) {
  const zs::CallRange range("zs_shard_step_accumulated_clipped");
  return zs::traced(zs_shard_step_accumulated_clipped_untraced(
                        plan, rank, lo, hi, grad_slices, grad_dtype, accum, micro_steps, master,
                        exp_avg, exp_avg_sq, full_flat, param_dtype, hp, step, coef, skip,
                        cuda_stream),
                    "zs_shard_step_accumulated_clipped", plan, rank, lo, hi, grad_dtype,
                    param_dtype, step);
}

extern "C" zs_status zs_grad_sqnorm_noalloc(const zs_plan* plan, int32_t rank, int64_t lo,
                                            int64_t hi, const void* const* grad_slices,
                                            zs_dtype grad_dtype, double* sqnorm_out,
                                            void* cuda_stream) {
  const zs::CallRange range("zs_grad_sqnorm_noalloc");
  return zs::traced(zs_grad_sqnorm_noalloc_untraced(plan, rank, lo, hi, grad_slices, grad_dtype,
                                                    sqnorm_out, cuda_stream),
                    "zs_grad_sqnorm_noalloc", plan, rank, lo, hi, grad_dtype, -1, 0);
}

extern "C" zs_status zs_clip_coefficient(const double* rank_sqnorms, int32_t n, double max_norm,
                                         float* coef_out, int32_t* nonfinite_out,
                                         void* cuda_stream) {
  const zs::CallRange range("zs_clip_coefficient");
  return zs::traced(zs_clip_coefficient_untraced(rank_sqnorms, n, max_norm, coef_out,
                                                 nonfinite_out, cuda_stream),
                    "zs_clip_coefficient", nullptr, -1, 0, 0, -1, -1, 0, n);
}

extern "C" zs_status zs_gather_assemble(const zs_plan* plan, int32_t rank,
                                        const void* const* shard_srcs, void* full_flat,
                                        zs_dtype param_dtype, void** views_out,
                                        void* cuda_stream) {
  const zs::CallRange range("zs_gather_assemble");
  return zs::traced(zs_gather_assemble_untraced(plan, rank, shard_srcs, full_flat, param_dtype,
                                                views_out, cuda_stream),
                    "zs_gather_assemble", plan, rank, 0, 0, -1, param_dtype, 0);
}

extern "C" zs_status zs_unshard(const zs_plan* plan, const void* gathered, zs_dtype dtype,
                                void* const* params_out, void* cuda_stream) {
  const zs::CallRange range("zs_unshard");
  return zs::traced(zs_unshard_untraced(plan, gathered, dtype, params_out, cuda_stream),
                    "zs_unshard", plan, -1, 0, 0, -1, dtype, 0);
}

extern "C" zs_status zs_shard_rows(const zs_plan* plan, int32_t rank, const void* const* params_in,
                                   zs_dtype dtype, void* local_out, void* cuda_stream) {
  const zs::CallRange range("zs_shard_rows");
  return zs::traced(zs_shard_rows_untraced(plan, rank, params_in, dtype, local_out, cuda_stream),
                    "zs_shard_rows", plan, rank, 0, 0, -1, dtype, 0);
}
