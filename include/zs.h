/*
 * zs.h — C ABI of the GB300 shard-local step for ZeRO-1/2/3 and FSDP.
 *
 * The step every data-parallel rank runs once the gradient ReduceScatter has
 * delivered its slices: sum the N incoming slices in fp32 and scale by 1/N,
 * run AdamW on this rank's fp32 master/m/v shard, cast the updated master to
 * the low-precision parameter straight into this rank's slot of the flat
 * buffer the parameter AllGather fills, and hand out per-tensor views of that
 * buffer. Pages followed (short names):
 *   [Dissection]  "ZeRO vs FSDP: A Rigorous Dissection for Distributed Training
 *                 Engineers"
 *   [Lifecycle]   "FSDP2's parameter lifecycle, and the wrap-policy bug that
 *                 turns one AllGather into ten"
 *   [DP-to-ZeRO]  "从 Data Parallel 到 ZeRO/FSDP：训练显存到底怎样被切开"
 *
 * Conventions for every call:
 *   - Returns zs_status: 0 on success, a negative code on error. No call
 *     aborts or exits; zs_last_error() gives a one-line detail (per thread).
 *   - Device buffers and CUDA streams are owned by the caller. The library
 *     allocates host memory for plans and pinned staging for the checkpoint
 *     calls (kept for the next one); it never allocates device memory.
 *   - Calls that take a stream enqueue work on it and return without
 *     synchronising (but for the checkpoint calls, which block); `cuda_stream`
 *     is a cudaStream_t (NULL = legacy default).
 *     Launch failures return ZS_ERR_CUDA.
 *   - Device pointers must be 16-byte aligned, resident on the current device,
 *     and (checked, where the driver can tell) cover the bytes the call uses;
 *     anything else is rejected before a kernel runs.
 */
#ifndef ZS_H
#define ZS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZS_MAX_WORLD 1024

typedef enum {
  ZS_OK = 0,
  ZS_ERR_INVAL = -1,       /* bad argument: NULL, unknown dtype, bad plan, overlap */
  ZS_ERR_ALIGN = -2,       /* a device pointer is not 16-byte aligned */
  ZS_ERR_RANGE = -3,       /* index range, rank or size out of bounds */
  ZS_ERR_CUDA = -4,        /* a CUDA runtime call or kernel launch failed */
  ZS_ERR_NOMEM = -5,       /* a host allocation failed (a plan, checkpoint staging) */
  ZS_ERR_TIMEOUT = -6,     /* a bounded device-side wait gave up */
  ZS_ERR_UNSUPPORTED = -7, /* combination not built into this library */
  ZS_ERR_IO = -8,          /* a checkpoint file could not be opened, read or written */
  ZS_ERR_CORRUPT = -9      /* a checkpoint file fails a check (format, size, checksum,
                              disagreement between the ranks' files) */
} zs_status;

/* Element types. ZS_FP24 is a 3-byte float: the top 24 bits of an fp32
 * pattern (sign, 8-bit exponent, 15-bit mantissa), rounded to nearest even,
 * stored little-endian. It exists only for the parameter-width sweep. */
typedef enum { ZS_BF16 = 0, ZS_FP32 = 1, ZS_FP24 = 2 } zs_dtype;

typedef struct zs_plan zs_plan; /* opaque, host memory, owned by the library */

typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
} zs_adamw_hparams;

/* ---------------------------------------------------------------------------
 * zs_flatten_plan — the flat-parameter layout and the rank shards.
 * [Dissection] §3.2 The FlatParameter Abstraction (concatenate a group's
 * parameters into one 1-D tensor; bookkeeping restores shapes);
 * [DP-to-ZeRO] "ZeRO Stage 1" (each rank owns about 1/N of the range);
 * [DP-to-ZeRO] "Shared Parameters 与 Tied Weights" (a shared weight has one
 * owner, flattened once); [DP-to-ZeRO] "ReduceScatter 必须尽早释放 Gradient"
 * (buckets ready in backward order).
 *
 *   numels[n_params]   element count of each parameter, registration order.
 *   tied_to[n_params]  -1 for a parameter with its own storage, or the index
 *                      k < i of the parameter it shares storage with (numels
 *                      must match); NULL = no ties.
 *   world              N, the number of data-parallel ranks (1..ZS_MAX_WORLD).
 *   align_elems        the padded total is a multiple of world*align_elems
 *                      (>= 1; 128 in the workloads).
 *   bucket_elems       0 = one bucket; else the greedy bucket limit in
 *                      elements (whole tensors, newest first).
 *   out                receives the plan; free it with zs_plan_free.
 * Layout: unique parameters back to back in registration order, no padding
 * between them; P = their total; P_pad = ceil(P / (N*align)) * N*align, the
 * tail [P, P_pad) is padding that holds zero in every buffer; S = P_pad / N;
 * rank r owns flat elements [r*S, (r+1)*S). The tail pad joins the bucket of
 * the last-registered tensor (bucket 0, the first ready).
 * Errors: ZS_ERR_INVAL (NULL, negative numel, bad tie), ZS_ERR_RANGE (world
 * or sizes out of range, int64 overflow), ZS_ERR_NOMEM.
 * ------------------------------------------------------------------------- */
zs_status zs_flatten_plan(const int64_t* numels, const int32_t* tied_to, int32_t n_params,
                          int32_t world, int64_t align_elems, int64_t bucket_elems,
                          zs_plan** out);

/* Plan queries. Any output pointer may be NULL. */
zs_status zs_plan_info(const zs_plan* plan, int64_t* P, int64_t* P_pad, int64_t* S,
                       int32_t* n_buckets, int32_t* world, int32_t* n_params);
/* offsets[n_params]: flat element offset of each parameter (a tied parameter
 * gets its owner's offset). */
zs_status zs_plan_offsets(const zs_plan* plan, int64_t* offsets, int32_t n_params);
/* Bucket b's flat range [flat_lo, flat_hi). */
zs_status zs_plan_bucket_range(const zs_plan* plan, int32_t bucket, int64_t* flat_lo,
                               int64_t* flat_hi);
/* Rank r's shard-local part [lo, hi) of bucket b (may be empty, lo == hi). */
zs_status zs_plan_bucket(const zs_plan* plan, int32_t bucket, int32_t rank, int64_t* lo,
                         int64_t* hi);
/* Frees a plan. Freeing a plan twice, or a pointer that is not a live plan,
 * returns ZS_ERR_INVAL and touches nothing. */
zs_status zs_plan_free(zs_plan* plan);

/* ---------------------------------------------------------------------------
 * zs_shard_step — the fused shard-local step of rank `rank` over shard-local
 * elements [lo, hi) (0, S = the whole shard; a bucket's part otherwise).
 * Reduce: [Dissection] §2.1 Mechanism and [Lifecycle] "The parameter
 * lifecycle": after the ReduceScatter each rank owns the reduced gradient of
 * its shard; [DP-to-ZeRO] "Data Parallel 保证的数学语义": that gradient is
 * the ranks' mean. Update: [DP-to-ZeRO] "ZeRO Stage 1" (the owner rank
 * updates its optimizer/parameter shard) with AdamW's fp32 master, m, v
 * ([Dissection] §1.1-1.2). Cast + place: [DP-to-ZeRO] "ZeRO Stage 1"
 * (all-gather the updated parameter shards) and "Mixed Precision 至少有四个
 * Dtype" (the master's low-precision copy).
 *
 * Per element i in [lo, hi), in fp32, each operation rounded to nearest even
 * and nothing fused:
 *   g   = (((0 + x_0[i]) + x_1[i]) + ... + x_{N-1}[i]) * fp32(1/N)
 *   m   = b1*m + (1-b1)*g;      v = b2*v + ((1-b2)*g)*g
 *   u   = (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps)
 *   p   = p*(1 - lr*wd) - lr*u;  full_flat[rank*S + i] = round(p)
 * with b1, b2, 1-b1, 1-b2, 1-b1^t, 1-b2^t, lr, eps, 1-lr*wd and 1/N each
 * computed once in double (beta^t by binary powering) and rounded to fp32.
 * One kernel launch: the register-streaming kernel or, for short ranges and
 * many slices, the staged kernel (zs_set_step_path); both compute exactly
 * these operations, so the result does not depend on which runs.
 *
 *   grad_slices[N]  device pointers; slice j is source rank j's gradient for
 *                   this rank's shard, element 0 of the shard at index 0,
 *                   S elements of grad_dtype (ZS_BF16 or ZS_FP32). Read only.
 *   master, exp_avg, exp_avg_sq
 *                   device fp32 [S], element 0 of the shard; updated in place.
 *   full_flat       device buffer of N*S elements of param_dtype; only
 *                   elements [rank*S + lo, rank*S + hi) are written.
 *   hp, step        AdamW hyper-parameters; step t >= 1 (bias correction).
 * The slices, the three state arrays and full_flat must not overlap one
 * another (slices may alias each other). Errors: ZS_ERR_INVAL (NULL, bad
 * plan, bad dtype, overlap, non-finite or out-of-range hyper-parameter),
 * ZS_ERR_ALIGN, ZS_ERR_RANGE (rank, lo/hi, step, a buffer shorter than its
 * extent), ZS_ERR_CUDA (launch failure).
 * ------------------------------------------------------------------------- */
zs_status zs_shard_step(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                        const void* const* grad_slices, zs_dtype grad_dtype, float* master,
                        float* exp_avg, float* exp_avg_sq, void* full_flat,
                        zs_dtype param_dtype, const zs_adamw_hparams* hp, int64_t step,
                        void* cuda_stream);

/* zs_shard_step with the cast parameters written into the rank's own
 * parameter shard instead of its slot of the flat buffer: param_shard is a
 * device buffer of S elements of param_dtype, element 0 of the shard at index
 * 0; elements [lo, hi) are written. For layouts that keep each rank's
 * parameters as a persistent shard of their own and all-gather them into a
 * transient buffer before use ([DP-to-ZeRO] "ZeRO 与 FSDP 的关系": FSDP2's
 * per-parameter sharded state; [Dissection] §2.3 ZeRO-3: each rank keeps 1/N
 * of the parameters). Same arithmetic, same kernels, same errors (param_shard
 * in the place of full_flat). */
zs_status zs_shard_step_to_shard(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                                 const void* const* grad_slices, zs_dtype grad_dtype,
                                 float* master, float* exp_avg, float* exp_avg_sq,
                                 void* param_shard, zs_dtype param_dtype,
                                 const zs_adamw_hparams* hp, int64_t step, void* cuda_stream);

/* ---------------------------------------------------------------------------
 * zs_gather_assemble — the AllGather's result on one GPU, and the unflatten.
 * [DP-to-ZeRO] "ZeRO Stage 1" (all-gather updated parameter shards; all
 * ranks again hold identical full parameters); [Dissection] §3.2 (the
 * bookkeeping that restores each parameter's view of the flat buffer).
 *
 *   shard_srcs[N]  device pointers to each rank's updated shard (S elements
 *                  of param_dtype). Entry `rank`, NULL entries, and entries
 *                  that already point at their own slot are skipped.
 *   full_flat      device buffer of N*S elements; slot j = [j*S, (j+1)*S)
 *                  receives shard_srcs[j] bit for bit.
 *   views_out      host array of n_params device pointers (may be NULL):
 *                  views_out[k] = full_flat + offsets[k]*elem_size; a tied
 *                  parameter gets its owner's pointer. Shapes are the caller's.
 * Errors as zs_shard_step; sources overlapping full_flat (other than their
 * own slot) are ZS_ERR_INVAL.
 * ------------------------------------------------------------------------- */
zs_status zs_gather_assemble(const zs_plan* plan, int32_t rank, const void* const* shard_srcs,
                             void* full_flat, zs_dtype param_dtype, void** views_out,
                             void* cuda_stream);

/* ---------------------------------------------------------------------------
 * Global-norm gradient clipping and the shared non-finite decision.
 * [DP-to-ZeRO] "Gradient Accumulation 会改变生命周期": a sharded step must
 * settle whether clipping uses the global norm or the local shard's, and
 * whether an overflow is decided by all ranks alike; its landing path checks
 * clipping by comparing single-step updates. Reading: the global L2 norm of
 * the reduced (mean) gradient; every rank skips the update when it is not
 * finite. Per step:
 *   1. each rank: zs_grad_sqnorm -> its shard's sum over i of g_i^2 (double);
 *   2. zs_clip_coefficient over the N partial sums (added in rank order; the
 *      scalar AllReduce of a real system) -> coef = fp32(min(1, max_norm /
 *      (sqrt(total) + 1e-6))) and nonfinite = !isfinite(sqrt(total));
 *   3. each rank: zs_shard_step_clipped with coef and nonfinite as `skip`.
 * Nothing returns to the host in between.
 * ------------------------------------------------------------------------- */

/* Bytes of scratch device memory zs_grad_sqnorm needs (1216 fp64 block
 * partials and a ticket word; 9984). The caller allocates and owns it. */
int64_t zs_grad_norm_workspace_bytes(void);

/* Sum over shard-local i in [lo, hi) of g_i^2, g_i the step's fp32 mean of the
 * N slices (same order and rounding as zs_shard_step), each square exact and
 * the sum carried in double; written to the device double *sqnorm_out. The
 * sum is reduced over a fixed 1216-block grid in a fixed order, so it is the
 * same on every run (it may differ from a sequential sum in the last bits).
 * workspace: 16-byte aligned device scratch of at least
 * zs_grad_norm_workspace_bytes() bytes, used by one call at a time. Errors as
 * zs_shard_step, plus ZS_ERR_RANGE for a short workspace. */
zs_status zs_grad_sqnorm(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                         const void* const* grad_slices, zs_dtype grad_dtype, void* workspace,
                         int64_t workspace_bytes, double* sqnorm_out, void* cuda_stream);

/* zs_grad_sqnorm for callers that cannot allocate device memory. The pages
 * have no counterpart to this call; it exists for this library's users. Some
 * callers cannot hand over scratch memory: code whose process has given the
 * whole device to another allocator that it cannot reach (a plug-in inside a
 * host application, say), or code that must still compute the gradient norm
 * after the device has run out of memory, to decide whether to skip the step
 * or to record why a rank is failing, when a cudaMalloc would itself fail.
 * This variant keeps the norm pass's scratch (1216 fp64 partials and a ticket
 * word, 9984 bytes: what one call needs whatever the input size, so every
 * call fits; the library is built only if the array holds it) in a static
 * device array of the library, held on every GPU that loads it until the
 * process exits. It calls no allocator. The caller still passes the inputs and
 * the output, as for zs_grad_sqnorm, and gets the same value, bit for bit. The
 * first call on a device looks the array up (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture. The address
 * is kept for the life of the process: do not use the library across a
 * cudaDeviceReset. All calls share the one array: calls that overlap on the
 * GPU (on different streams, or from several threads) race and must not be
 * issued; calls in order on one stream are safe, each clearing what must
 * start at zero. */
zs_status zs_grad_sqnorm_noalloc(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                                 const void* const* grad_slices, zs_dtype grad_dtype,
                                 double* sqnorm_out, void* cuda_stream);

/* rank_sqnorms: device double [n], the ranks' partial sums (1 <= n <= 1024).
 * Writes the device fp32 *coef_out and the device int32 *nonfinite_out (1 when
 * the global norm is Inf or NaN; coef is then 1). max_norm: finite, > 0. */
zs_status zs_clip_coefficient(const double* rank_sqnorms, int32_t n, double max_norm,
                              float* coef_out, int32_t* nonfinite_out, void* cuda_stream);

/* zs_shard_step with g = (mean) * (*coef) when coef is not NULL, and no change
 * to any buffer when skip is not NULL and *skip != 0. coef and skip are device
 * pointers read by the kernel (4-byte aligned). With coef == NULL and skip ==
 * NULL it is zs_shard_step. */
zs_status zs_shard_step_clipped(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                                const void* const* grad_slices, zs_dtype grad_dtype,
                                float* master, float* exp_avg, float* exp_avg_sq,
                                void* full_flat, zs_dtype param_dtype,
                                const zs_adamw_hparams* hp, int64_t step, const float* coef,
                                const int32_t* skip, void* cuda_stream);

/* ---------------------------------------------------------------------------
 * Gradient accumulation on the shard (G micro-batches per optimizer step).
 * [DP-to-ZeRO] "Gradient Accumulation 会改变生命周期": whether each micro-step
 * ReduceScatters, whether to accumulate on the shard or the full tensor, and
 * whether the loss is divided by G must be decided; [Dissection] §7 (gradient
 * accumulation). Reading: every micro-step ReduceScatters (ZeRO-2/3: no rank
 * holds a full gradient); the mean of the micro-step's N slices is added into
 * an fp32 accumulator of the shard; the last micro-step's slices go straight
 * into the step, which uses ((accumulator + mean) * fp32(1/G)), the average
 * over the G micro-batches (equivalently, the loss divided by G).
 *   micro-steps 1 .. G-1: zs_grad_accumulate (first = 1 on micro-step 1, which
 *                         overwrites the accumulator instead of adding);
 *   micro-step G:         zs_shard_step_accumulated.
 * ------------------------------------------------------------------------- */

/* accum[i] = (first ? 0 : accum[i]) + mean_j x_j[i] for shard-local i in
 * [lo, hi), the mean formed as zs_shard_step forms it (fp32, j ascending,
 * times fp32(1/N)). accum: device fp32 [S], element 0 of the shard, must not
 * overlap the slices. Errors as zs_shard_step. */
zs_status zs_grad_accumulate(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                             const void* const* grad_slices, zs_dtype grad_dtype, float* accum,
                             int32_t first, void* cuda_stream);

/* zs_shard_step on g = (accum[i] + mean_j x_j[i]) * fp32(1/micro_steps), with
 * accum (device fp32 [S], read only) holding the sum of the earlier
 * micro-steps' means. micro_steps >= 1; accum must not overlap any output. */
zs_status zs_shard_step_accumulated(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                                    const void* const* grad_slices, zs_dtype grad_dtype,
                                    const float* accum, int32_t micro_steps, float* master,
                                    float* exp_avg, float* exp_avg_sq, void* full_flat,
                                    zs_dtype param_dtype, const zs_adamw_hparams* hp,
                                    int64_t step, void* cuda_stream);

/* Clipping an accumulated gradient (both questions of the section above at
 * once). The clip acts on the gradient the update sees, the micro-batch
 * average g = (accum + mean) * fp32(1/G): its global norm, not the last
 * micro-step's, decides the coefficient. Per optimizer step, after micro-steps
 * 1 .. G-1 went through zs_grad_accumulate:
 *   1. each rank: zs_grad_sqnorm_accumulated -> its shard's sum of g_i^2;
 *   2. zs_clip_coefficient over the N partial sums, as for the plain step;
 *   3. each rank: zs_shard_step_accumulated_clipped with coef and skip.
 *
 * zs_grad_sqnorm with g_i = (accum[i] + mean_j x_j[i]) * fp32(1/micro_steps),
 * formed as zs_shard_step_accumulated forms it. accum: device fp32 [S], read
 * only. Errors as zs_grad_sqnorm and zs_shard_step_accumulated. */
zs_status zs_grad_sqnorm_accumulated(const zs_plan* plan, int32_t rank, int64_t lo, int64_t hi,
                                     const void* const* grad_slices, zs_dtype grad_dtype,
                                     const float* accum, int32_t micro_steps, void* workspace,
                                     int64_t workspace_bytes, double* sqnorm_out,
                                     void* cuda_stream);
/* zs_shard_step_accumulated on g * (*coef) (coef NULL: no scaling), and no
 * change to any buffer when skip is not NULL and *skip != 0; coef and skip as
 * in zs_shard_step_clipped. With coef == skip == NULL it is
 * zs_shard_step_accumulated. */
zs_status zs_shard_step_accumulated_clipped(const zs_plan* plan, int32_t rank, int64_t lo,
                                            int64_t hi, const void* const* grad_slices,
                                            zs_dtype grad_dtype, const float* accum,
                                            int32_t micro_steps, float* master, float* exp_avg,
                                            float* exp_avg_sq, void* full_flat,
                                            zs_dtype param_dtype, const zs_adamw_hparams* hp,
                                            int64_t step, const float* coef,
                                            const int32_t* skip, void* cuda_stream);

/* ---------------------------------------------------------------------------
 * Per-parameter row sharding (FSDP2) and the gather side of a wrap unit.
 * [DP-to-ZeRO] "ZeRO 与 FSDP 的关系": FSDP2's fully_shard keeps per-parameter
 * sharded state and unshards before forward/backward, reshards after;
 * [Lifecycle] "The parameter lifecycle, one module at a time" and "Reshard
 * policy": AllGather before a module's compute, then reshard to 1/N, retain,
 * or (an integer reshard_after_forward) reshard to a smaller world.
 * Layout of a row-sharded plan: parameter i (dim0 rows of numel/dim0
 * elements) is cut along dim 0 into N chunks of c_i = ceil(dim0/N) rows;
 * rank r holds rows [r*c_i, min((r+1)*c_i, dim0)) (possibly none) padded with
 * zero rows to c_i; a rank's local buffer is its padded chunks back to back in
 * registration order (tied parameters once), zero-padded at the end to a
 * multiple of align_elems: S elements. zs_plan_info reports S, P (the unique
 * elements) and P_pad = N*S, the rank-major AllGather buffer. zs_shard_step
 * and zs_gather_assemble work on these plans unchanged (S is a rank's shard);
 * the gathered buffer is copied out into parameters by zs_unshard.
 * ------------------------------------------------------------------------- */
zs_status zs_rows_plan(const int64_t* dim0, const int64_t* numels, const int32_t* tied_to,
                       int32_t n_params, int32_t world, int64_t align_elems, zs_plan** out);
/* rows_per_rank[i] = c_i and row_elems[i] = numel/dim0 (either may be NULL);
 * zs_plan_offsets gives each parameter's segment offset in a local buffer. */
zs_status zs_plan_rows(const zs_plan* plan, int64_t* rows_per_rank, int64_t* row_elems,
                       int32_t n_params);
/* Copy-out of the AllGather: gathered = [N][S] elements of dtype, rank-major;
 * params_out[i] = device pointer to parameter i's full tensor (numel_i
 * elements, contiguous; entries of tied parameters are ignored). Writes every
 * row of every owner parameter. Row-sharded plans only (ZS_ERR_UNSUPPORTED
 * otherwise). */
zs_status zs_unshard(const zs_plan* plan, const void* gathered, zs_dtype dtype,
                     void* const* params_out, void* cuda_stream);
/* Copy-in / reshard: rank `rank`'s local buffer (S elements of dtype) from the
 * full parameters, padding zeroed. With a plan made for a smaller world M this
 * is reshard_after_forward = M. Row-sharded plans only. */
zs_status zs_shard_rows(const zs_plan* plan, int32_t rank, const void* const* params_in,
                        zs_dtype dtype, void* local_out, void* cuda_stream);

/* -------------------------------------------------------------------------
 * Sharded checkpoint and resharding restore. [DP-to-ZeRO] "Checkpoint 不能假设
 * 每个 Rank 都有完整模型": with sharded state each rank saves its own shards
 * plus the metadata that places them in the global tensors; a restore into
 * another world size reshards; a consistent checkpoint holds the master
 * weights, the optimizer moments, the global step and the sharding metadata;
 * and a restore is right only when the next update equals that of the
 * uninterrupted run (its "常见误区" section). Its landing path, step 10: save,
 * fault injection, restore at the same and at another world size.
 *
 * One file per rank holds: a header (format version, layout, world, rank,
 * P, S, step), the parameter list with the plan's layout, the fp32 master /
 * exp_avg / exp_avg_sq shard (S elements each), and a 64-bit checksum per
 * 1 MiB block of each array. Element e of parameter i has one place in the
 * global tensor in every layout, so a file saved under one plan loads into
 * any plan over the same parameter list (numels and ties equal): another
 * world size, and flat <-> row layouts. The new shard's padding is zeroed.
 *
 * State arrays are all device memory (current device, 16-byte aligned) or
 * all host memory. Device-resident state moves through pinned host staging
 * (three 64 MiB buffers; no device memory is allocated). The first call on
 * device state allocates the staging and the library keeps one set for the
 * next call on the same device, until zs_checkpoint_release_staging; saving
 * hashes the blocks on the device, and so does loading for
 * every block that lands whole in the device arrays. Both calls block until
 * done, enqueueing their device work on `cuda_stream` and synchronising it.
 * Not thread-safe for one path. Errors: ZS_ERR_IO (open/read/write),
 * ZS_ERR_CORRUPT (bad magic or version, header or metadata checksum, file
 * size, block checksum, files of different steps or layouts, a file in the
 * wrong rank's place), ZS_ERR_INVAL (the parameter list differs from the
 * plan's, NULL arguments, mixed host/device arrays).
 * ------------------------------------------------------------------------- */
/* Writes rank `rank`'s shard of `plan` (S fp32 elements per array) and `step`
 * to `path`, through `path` + ".part" renamed on success (no torn file under
 * the final name; the file is not fsync'ed). */
zs_status zs_checkpoint_save(const zs_plan* plan, int32_t rank, const float* master,
                             const float* exp_avg, const float* exp_avg_sq, int64_t step,
                             const char* path, void* cuda_stream);
/* Fills rank `rank`'s shard of `plan` from the files saved by the old ranks:
 * paths[k] = old rank k's file, n_paths = the old world. Entries of old ranks
 * whose elements this rank does not hold may be NULL (paths[0] never: it fixes
 * the old layout). Every block read is checked against its checksum (on the
 * device after it lands, or on the host before it is copied); on
 * ZS_ERR_CORRUPT / ZS_ERR_IO the arrays may hold partial data. *step = the
 * saved step (may be NULL). */
zs_status zs_checkpoint_load(const zs_plan* plan, int32_t rank, const char* const* paths,
                             int32_t n_paths, float* master, float* exp_avg, float* exp_avg_sq,
                             int64_t* step, void* cuda_stream);
/* Frees the pinned staging the checkpoint calls keep between calls (none
 * kept: nothing to do). Not to be called while a checkpoint call runs. */
zs_status zs_checkpoint_release_staging(void);
/* The header of a checkpoint file, checked (any output may be NULL). layout:
 * 0 flat, 1 rows. */
zs_status zs_checkpoint_info(const char* path, int32_t* world, int32_t* rank, int32_t* layout,
                             int32_t* n_params, int64_t* P, int64_t* S, int64_t* step);

/* -------------------------------------------------------------------------
 * Per-call trace. [DP-to-ZeRO] "训练 Hang 应按 Collective 顺序排查": ZeRO/FSDP
 * issue their collectives from hooks, so ranks that run modules in another
 * order or another number of times end up waiting in different collectives;
 * the section's remedy is to log, for each collective, its sequence number,
 * group, numel, dtype, module and phase, and look for the first place where
 * the ranks' logs part.
 *
 * Each call that stands at a collective of the real system (the steps, the
 * accumulation, the norm and the clip coefficient, the gather assembly, the
 * row copy-out and copy-in, checkpoint save and load) appends one line to
 * this process's trace when tracing is on, after it returns:
 *   seq=<n> call=<name> plan=<id> world=<N> S=<shard elements> rank=<r>
 *   lo=<lo> hi=<hi> grad=<dtype> param=<dtype> step=<t> status=<code>
 * seq counts from 0 per trace file; plan is a 64-bit hash of the plan's
 * parameter list and layout ("-" when the call has no live plan); dtypes are
 * bf16 / fp32 / fp24 or "-". Tracing is off until ZS_TRACE names a file
 * (read at the first traced call) or zs_set_trace is called; in the name, %r
 * stands for the RANK environment variable (0 if unset) and %p for the
 * process id. Lines are appended under a lock and flushed per record. The
 * pages have no device-side counterpart; this is the host log they ask for.
 * ------------------------------------------------------------------------- */
/* Opens `path` (expanded as above, appended to) as this process's trace and
 * restarts seq at 0; NULL or "" turns tracing off (and ZS_TRACE is not read
 * afterwards). ZS_ERR_IO if the file cannot be opened (tracing is then off). */
zs_status zs_set_trace(const char* path);
/* Compares the traces of the ranks of one job record by record on the fields
 * all ranks must share at one seq (call, plan, world, S, grad, param, step;
 * not rank, lo, hi, status) and reports the first seq at which they differ,
 * or at which a trace ends while another goes on: *seq_out = that seq, or -1
 * when all agree to the end. `detail` (if not NULL, `detail_bytes` long)
 * receives the differing records, one per trace, NUL-terminated and cut to
 * fit. n_paths >= 2. ZS_ERR_IO if a file cannot be read. */
zs_status zs_trace_first_divergence(const char* const* paths, int32_t n_paths, int64_t* seq_out,
                                    char* detail, int64_t detail_bytes);

/* Diagnostics. */
const char* zs_status_string(zs_status status);
const char* zs_last_error(void);
/* Synchronises `cuda_stream`, then reads and clears this device's error word
 * (set by the bounds-checked build's checks and by bounded waits);
 * ZS_ERR_TIMEOUT or ZS_ERR_RANGE if it was set, ZS_ERR_CUDA if the stream
 * reports an error. The library looks the addresses of its device arrays
 * (this error word, the no-alloc norm scratch) up once per device and keeps
 * them for the life of the process: it is not to be used across a
 * cudaDeviceReset of a device it has used. */
zs_status zs_check_device_error(void* cuda_stream);
/* The bounds-checked build. The library also exists as libzs_checked.so: the
 * same host code, and kernels that check, before each global access or bulk
 * copy, that what it touches lies in the window its launch declares (the
 * shard range [lo, hi) for the step, accumulation and norm kernels; the slot
 * and the world's buffer for the gather; the segment for the row copies; the
 * block for the checksums). A range outside its window is not accessed and
 * sets the error word's bounds bit (ZS_ERR_RANGE from zs_check_device_error);
 * no trap, the context stays usable. For tests of the kernels' index
 * arithmetic, not for timing. Returns 1 in that build, else 0. The pages have
 * no counterpart (their tooling stops at profilers). */
int32_t zs_bounds_checked(void);
/* Checked build only: narrows the window of the step, accumulation and norm
 * kernels to [lo + shrink, hi - shrink) (0 = the range itself), so that a
 * test sees the checks fire on accesses that are in fact in bounds. Process-
 * wide. ZS_ERR_UNSUPPORTED in the ordinary build, ZS_ERR_RANGE for shrink
 * outside 0..2^40. */
zs_status zs_selftest_bounds_window(int64_t shrink);
/* The step's kernel. Two kernels compute the same step with the same fp32
 * operations in the same order (results are identical): the register-
 * streaming kernel (each thread loads its 16-element group of every slice and
 * state array straight into registers) and the staged kernel (one or two
 * blocks per SM; one warp streams 2048- or 1024-element tiles of the slices
 * and state into shared memory with bulk asynchronous copies while 16 warps
 * compute;
 * where two stages fit: N <= 50 bf16 or 25 fp32 slices). path 0 (default):
 * chosen per call by N, the slice and parameter dtypes and the range's
 * length (mostly the staged kernel); 1: always the register-streaming
 * kernel; 2: the staged kernel wherever it applies.
 * Returns the previous path, or -1 for an unknown path (nothing changed).
 * The pages have no counterpart: this is a choice between two GB300 kernels. */
int32_t zs_set_step_path(int32_t path);
/* 1 (default): the library's kernels are launched so that each may be
 * scheduled while the previous kernel in its stream finishes (programmatic
 * dependent launch); every kernel waits, before its first access to global
 * memory, until the kernels before it have completed and their writes are
 * visible, so stream order and results are those of ordinary launches. This
 * hides most of a launch's ramp between back-to-back calls (a bucket's step
 * after another's, the norm pass, coefficient and clipped step). 0: ordinary
 * launches. Process-wide; returns the previous setting, or -1 for a value
 * other than 0 or 1 (nothing changed). The pages have no counterpart: this is
 * how the GPU schedules this library's launches. */
int32_t zs_set_launch_overlap(int32_t on);
/* Which kernel ran the calling thread's last step-family launch (zs_shard_step
 * and its clipped, accumulated and to-shard forms): *kernel = 1 for the
 * register-streaming kernel, with *elems = the elements of one thread's vector
 * group (16: 32-byte accesses, 8: 16-byte accesses, 0: element by element);
 * *kernel = 2 for the staged kernel, with *elems = the elements of one tile
 * (2048 or 1024). *kernel = 0 and *elems = 0 before the thread's first launch.
 * A call that launches nothing (an empty range, an argument error, a launch
 * that fails) leaves the record as it was. For tests that must know which code path a call took; the pages
 * have no counterpart. ZS_ERR_INVAL for NULL outputs. */
zs_status zs_last_step_kernel(int32_t* kernel, int32_t* elems);
/* Failure detection without a fault: enqueues one block that waits, through
 * the same bounded mbarrier wait the staged step kernel uses, on a barrier
 * nothing arrives on, giving up after `polls` polls (1..2^20). The wait then
 * sets the device error word's timeout bit, so a following
 * zs_check_device_error returns ZS_ERR_TIMEOUT; the context stays usable.
 * The pages have no counterpart (their failure detection is watchdog
 * timeouts on hung collectives). */
zs_status zs_selftest_wait_timeout(uint32_t polls, void* cuda_stream);
/* 1 = check device pointers against the driver's allocation records on each
 * call (default), 0 = only NULL/alignment/range checks. Returns the old level. */
int32_t zs_set_validation(int32_t level);
/* Library version, "major.minor.patch". */
const char* zs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZS_H */
