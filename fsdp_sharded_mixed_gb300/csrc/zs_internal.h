// zs_internal.h — declarations shared by the library's own translation units
// (planner, C-ABI layer, kernels). Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/zs.h"

struct zs_plan {
  uint64_t magic;
  int32_t layout;      // kLayoutFlat (one flat buffer cut into N pieces) or kLayoutRows
  int32_t world;
  int32_t n_params;
  int64_t align;
  int64_t bucket_elems;
  int64_t P, P_pad, S;
  std::vector<int64_t> numels;
  std::vector<int64_t> offsets;
  std::vector<int32_t> owner;
  std::vector<int64_t> bucket_lo, bucket_hi;
  // kLayoutRows: dim0[i] rows of row_elems[i] elements; rows_per_rank[i] =
  // ceil(dim0 / N); offsets[i] = the parameter's segment offset inside every
  // rank's local buffer (S elements, the segments back to back, padded).
  std::vector<int64_t> dim0, row_elems, rows_per_rank;
};

namespace zs {

constexpr int32_t kLayoutFlat = 0;
constexpr int32_t kLayoutRows = 1;
constexpr uint64_t kPlanMagic = 0x7A735F706C616E31ull;  // "zs_plan1"

// Thread-local error detail; returns `st` so call sites can `return fail(...)`.
zs_status fail(zs_status st, const char* fmt, ...);
void clear_error();

// True when `plan` is a live plan made by zs_flatten_plan.
bool plan_is_live(const zs_plan* plan);

// fp32 scalars of one optimizer step, computed on the host from doubles.
struct StepScalars {
  float b1, b2, omb1, omb2, bc1, bc2, lr, eps, decay, invN;
};

// The index window a kernel's accesses are checked against in the bounds-
// checked build (the CUDA sources compiled with ZS_BOUNDS_CHECK=1, see
// bounds.cuh): [lo, hi) in elements of the shard. Every build carries it in
// the launch structures; only the checked build's kernels read it.
struct Window {
  int64_t lo, hi;
};
// The step-family window for the range [lo, hi): the range itself, narrowed
// at both ends by the self-test shrink (zs_selftest_bounds_window).
Window step_window(int64_t lo, int64_t hi);
// 1 in the bounds-checked build, 0 otherwise (defined by the CUDA sources).
int bounds_checked();

// Kernel launchers (shard_step.cu, gather.cu). They assume validated input.
struct ShardStepLaunch {
  const void* const* grads;  // host array of N device pointers
  int32_t world;
  zs_dtype grad_dtype, param_dtype;
  float* master;
  float* m;
  float* v;
  unsigned char* slot;  // full_flat + rank*S*elem_bytes
  int64_t lo, hi;
  int vec_width;        // elements per vector group: 16 (32-byte accesses),
                        // 8 (16-byte accesses) or 0 (element by element)
  const float* coef;    // device fp32 clip coefficient, or NULL (no clipping)
  const int32_t* skip;  // device flag: non-zero leaves every buffer as it is, or NULL
  const float* accum;   // fp32 [S] micro-step accumulator (accumulation kernels), or NULL
  float invG;           // fp32(1/G) for the accumulated step
  StepScalars s;
  Window win;           // checked build: every element the kernels touch lies in it
};
cudaError_t launch_shard_step(const ShardStepLaunch& a, cudaStream_t stream);
// Gradient accumulation (accum.cu): accum = (first ? 0 : accum) + mean, and the
// step on ((accum + mean) * invG).
cudaError_t launch_grad_accumulate(const ShardStepLaunch& a, int first, cudaStream_t stream);
cudaError_t launch_shard_step_accumulated(const ShardStepLaunch& a, cudaStream_t stream);

struct GatherLaunch {
  const unsigned char* const* srcs;  // host array of N pointers (NULL = skip)
  int32_t world;
  unsigned char* dst;                // full_flat
  int64_t slot_bytes;
};
cudaError_t launch_gather(const GatherLaunch& a, cudaStream_t stream);

// Global-norm pass (clip.cu): per-block partial sums of squares in scratch
// memory, reduced in block order by the last block.
constexpr int kNormPartials = 1216;  // 8 x 152 SMs
constexpr int64_t kNormTicketOffset = kNormPartials * 8;   // bytes
constexpr int64_t kNormWorkspaceBytes = kNormTicketOffset + 256;
struct NormLaunch {
  const void* const* grads;
  int32_t world;
  zs_dtype grad_dtype;
  int64_t lo, hi;
  bool vec;             // all slices 32-byte aligned: 16-element vector groups
  float invN;
  double* partials;     // [kNormPartials]
  unsigned int* ticket;
  double* out;
  Window win;           // checked build: every element the pass reads lies in it
  const float* accum;   // fp32 [S] accumulator: the norm of (accum + mean) * invG; or NULL
  float invG;           // fp32(1/G) with accum
};
cudaError_t launch_grad_sqnorm(const NormLaunch& a, cudaStream_t stream);
// The same norm pass with its scratch in a file-scope device array of
// kNoAllocScratchBytes (clip.cu); callers check kNormWorkspaceBytes fits.
constexpr int64_t kNoAllocScratchBytes = 9984;
cudaError_t launch_grad_sqnorm_noalloc(const NormLaunch& a, cudaStream_t stream);
cudaError_t launch_clip_coef(const double* rank_sqnorms, int n, double max_norm, float* coef,
                             int32_t* nonfinite, cudaStream_t stream);

// Segment copies of the row-sharded layout (rows.cu): copy_bytes from src to
// dst, then zero_bytes of zeros after them at dst.
struct RowSegment {
  const unsigned char* src;
  unsigned char* dst;
  int64_t copy_bytes;
  int64_t zero_bytes;
};
constexpr int kMaxSegs = 256;
cudaError_t launch_segment_copy(const RowSegment* segs, int n, cudaStream_t stream);

// Block checksums of checkpoint data (ckpt.cu, definition in block_hash.h):
// the checksum of bytes [j*block_bytes, min((j+1)*block_bytes, bytes)) of
// `data` (16-byte aligned) as block first_block + j of array `array_id` is
// the sum (mod 2^64) of out[j*parts + p], p < parts. block_hash_parts gives
// the parts (a power of two) that spread `blocks` blocks over every SM.
cudaError_t launch_block_hash(const void* data, int64_t bytes, int64_t first_block,
                              int64_t block_bytes, uint32_t array_id, int parts, uint64_t* out,
                              cudaStream_t stream);
int block_hash_parts(int64_t blocks, int64_t block_bytes);

// Argument checks of the C-ABI layer, for the other host translation units:
// device-resident on the current device and (where the driver can tell)
// [p, p + bytes) inside one allocation.
zs_status check_device_array(const void* p, int64_t bytes, const char* fn, const char* name);

// Appends one record of a call to the per-call trace when tracing is on
// (trace.cpp) and returns st. grad_dtype / param_dtype -1 = not applicable;
// world is used when plan is not a live plan.
zs_status traced(zs_status st, const char* call, const zs_plan* plan, int32_t rank, int64_t lo,
                 int64_t hi, int grad_dtype, int param_dtype, int64_t step, int32_t world = 0);

// An NVTX range named after a library call, open for the object's lifetime,
// so that profilers attribute the call's host time and launches to it. NVTX
// costs a pointer test per call when no tool is attached.
class CallRange {
 public:
  explicit CallRange(const char* name);
  ~CallRange();
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

// Which kernel runs the step: 0 = chosen per call, 1 = the register-streaming
// kernel, 2 = the staged kernel wherever it is eligible (zs_set_step_path).
int step_path();
// Records, for zs_last_step_kernel, the kernel the calling thread's step-family
// launch used: 1 = register-streaming (elems = vector group: 16, 8, 0),
// 2 = staged (elems = tile elements).
void note_step_kernel(int kernel, int elems);
// This device's error word (device address), for kernels that report into it.
unsigned int* device_error_word();
// One block waiting, bounded by `polls`, on an mbarrier nothing arrives on.
cudaError_t launch_wait_timeout(uint32_t polls, cudaStream_t stream);

// Device error word: bit value 1 set by the bounds-checked build's checks,
// 2 by bounded waits that gave up.
cudaError_t read_and_clear_device_error(cudaStream_t stream, unsigned int* word);

int elem_bytes(zs_dtype dt);

}  // namespace zs
