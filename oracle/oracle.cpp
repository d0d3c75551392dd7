/*
 * oracle.cpp — CPU oracle for the ZeRO/FSDP shard-local step.
 *
 * TEST INFRASTRUCTURE. This is a plain, slow, single-threaded restatement of
 * what the shard-local step computes, used only to check the CUDA path. Only
 * the tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code with the CUDA path (no headers, helpers or tables), and the
 * product library never calls it.
 *
 * Build: g++ -std=c++17 -O2 -ffp-contract=off (no -ffast-math), so that every
 * float operation below is one IEEE-754 binary32 operation rounded to nearest
 * even, sqrtf is the correctly rounded square root, and nothing is fused.
 *
 * Pages cited (short names used below):
 *   [Dissection]  "ZeRO vs FSDP: A Rigorous Dissection for Distributed Training
 *                 Engineers" (fp4-site.pages.dev)
 *   [Lifecycle]   "FSDP2's parameter lifecycle, and the wrap-policy bug that
 *                 turns one AllGather into ten" (deepnotes.pages.dev)
 *   [DP-to-ZeRO]  "从 Data Parallel 到 ZeRO/FSDP：训练显存到底怎样被切开"
 *                 (charlestar.github.io)
 *   [Measured]    "DeepSpeed ZeRO vs PyTorch FSDP2, measured" (dev.to)
 *
 * The pages name AdamW and its three fp32 states but print no update
 * equations; the update below is Adam (Kingma & Ba, ICLR 2015, Algorithm 1)
 * with decoupled weight decay (Loshchilov & Hutter, ICLR 2019, Algorithm 2),
 * the decay scaled by the learning rate. Its exact rounding sequence is a
 * reading, not something the pages fix: that part is pinned only by the
 * closed forms and invariants in the tests (parity of the rounding sequence
 * itself is unpinned by the pages).
 */
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

enum : int32_t { DT_BF16 = 0, DT_FP32 = 1, DT_FP24 = 2 };

int elem_bytes(int32_t dt) {
  switch (dt) {
    case DT_BF16: return 2;
    case DT_FP32: return 4;
    case DT_FP24: return 3;
    default: return 0;
  }
}

uint32_t float_bits(float x) {
  uint32_t b;
  std::memcpy(&b, &x, 4);
  return b;
}

float bits_float(uint32_t b) {
  float x;
  std::memcpy(&x, &b, 4);
  return x;
}

/* bf16 -> fp32 widening: a bf16 value is the top half of an fp32 pattern, so
 * the widening is exact. */
float bf16_to_float(uint16_t h) { return bits_float((uint32_t)h << 16); }

/* Round an fp32 value to the nearest value whose low `drop` mantissa bits are
 * zero, ties to the one whose lowest kept bit is 0 (round-to-nearest-even),
 * and return the kept high bits. NaN becomes the canonical quiet NaN of the
 * narrow format with the input's sign. Overflow rounds to infinity through
 * the carry into the exponent, as nearest-even rounding requires. Subnormals
 * are rounded like any other pattern (no flush to zero). */
uint32_t round_keep_high(float x, int drop) {
  uint32_t b = float_bits(x);
  uint32_t sign = b & 0x80000000u;
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu) != 0u)
    return (sign | 0x7FC00000u) >> drop;
  uint32_t half = 1u << (drop - 1);
  uint32_t low = b & ((1u << drop) - 1u);
  uint32_t keep = b >> drop;
  if (low > half || (low == half && (keep & 1u))) keep += 1u;
  return keep;
}

/* The optimizer step's fp32 scalars, computed once per step from doubles and
 * rounded to fp32 once each. beta^t is the right-to-left binary powering
 * (Knuth, TAOCP vol. 2, 4.6.3, Algorithm A) in IEEE double. */
struct Scalars {
  float b1, b2, omb1, omb2, bc1, bc2, lr, eps, decay, invN;
};

double power_by_squaring(double base, int64_t e) {
  double result = 1.0;
  while (e > 0) {
    if (e & 1) result = result * base;
    base = base * base;
    e >>= 1;
  }
  return result;
}

Scalars make_scalars(double lr, double beta1, double beta2, double eps, double wd,
                     int64_t t, int32_t world) {
  Scalars s;
  s.b1 = (float)beta1;
  s.b2 = (float)beta2;
  s.omb1 = (float)(1.0 - beta1);
  s.omb2 = (float)(1.0 - beta2);
  s.bc1 = (float)(1.0 - power_by_squaring(beta1, t));
  s.bc2 = (float)(1.0 - power_by_squaring(beta2, t));
  s.lr = (float)lr;
  s.eps = (float)eps;
  s.decay = (float)(1.0 - lr * wd);
  s.invN = (float)(1.0 / (double)world);
  return s;
}

/* One element of AdamW on the fp32 master/m/v shard.
 * Adam moments and bias correction (Kingma & Ba, Alg. 1), then the decoupled
 * decay theta*(1 - lr*wd) applied to the previous master value together with
 * the Adam step (Loshchilov & Hutter, Alg. 2). The three fp32 states are the
 * 12 optimizer bytes of [Dissection] §1.1-1.2 and [Lifecycle] "16 bytes per
 * parameter is where planning starts". Each line is one rounded fp32 op. */
void adamw_element(const Scalars& s, float g, float& p, float& m, float& v) {
  float m_prev_term = s.b1 * m;
  float g_term = s.omb1 * g;
  m = m_prev_term + g_term;

  float v_prev_term = s.b2 * v;
  float g_scaled = s.omb2 * g;
  float g_sq_term = g_scaled * g;
  v = v_prev_term + g_sq_term;

  float m_hat = m / s.bc1;
  float v_hat = v / s.bc2;
  float denom = std::sqrt(v_hat) + s.eps;
  float update = m_hat / denom;

  float decayed = p * s.decay;
  float step = s.lr * update;
  p = decayed - step;
}

float load_grad(const void* base, int32_t dt, int64_t i) {
  if (dt == DT_BF16) return bf16_to_float(static_cast<const uint16_t*>(base)[i]);
  return static_cast<const float*>(base)[i];
}

/* Store the low-precision parameter (the mixed-precision cast of the master,
 * [DP-to-ZeRO] "Mixed Precision 至少有四个 Dtype"). bf16 and the 3-byte
 * variant are nearest-even roundings of the fp32 master; fp32 is a copy. The
 * 3-byte variant is stored little-endian. */
void store_param(void* base, int32_t dt, int64_t i, float p) {
  if (dt == DT_BF16) {
    static_cast<uint16_t*>(base)[i] = (uint16_t)round_keep_high(p, 16);
  } else if (dt == DT_FP32) {
    static_cast<float*>(base)[i] = p;
  } else {
    uint32_t q = round_keep_high(p, 8);
    uint8_t* d = static_cast<uint8_t*>(base) + 3 * i;
    d[0] = (uint8_t)(q & 0xFFu);
    d[1] = (uint8_t)((q >> 8) & 0xFFu);
    d[2] = (uint8_t)((q >> 16) & 0xFFu);
  }
}

}  // namespace

extern "C" {

/* ---------------------------------------------------------------------------
 * O1. Flatten plan.
 * [Dissection] §3.2 The FlatParameter Abstraction: a group's parameters are
 * concatenated into one 1-D tensor, with bookkeeping to restore the shapes.
 * [DP-to-ZeRO] "ZeRO Stage 1": each rank updates about 1/N of the parameter
 * range (contiguous rank shards). [DP-to-ZeRO] "一次 Mixed-precision Adam…":
 * padding/flattening/alignment add bytes; tied weights affect deduplication.
 * [DP-to-ZeRO] "Shared Parameters 与 Tied Weights": a shared weight has one
 * owner and is flattened once.
 * [DP-to-ZeRO] "ReduceScatter 必须尽早释放 Gradient": buckets become ready in
 * backward order, i.e. reverse registration order, and are made of whole
 * parameters.
 *
 * Readings: unique parameters are concatenated in registration order with no
 * padding between them; the total is padded with zeros to a multiple of
 * world*align; rank r owns [r*S, (r+1)*S). Buckets are formed greedily over
 * unique parameters in reverse registration order; a bucket closes when the
 * next tensor would push it past bucket_elems; a tensor is never split; the
 * tail pad joins the bucket holding the last-registered tensor.
 *
 * tied_to[i] = -1 for an owner, or the index k < i of the parameter it shares
 * storage with (chains resolve to the first owner; numels must match).
 * Outputs: offsets[n_params] (tied -> owner's offset), info = {P, P_pad, S,
 * n_buckets}, bucket_lo/hi = flat ranges in bucket order (first ready first).
 * Returns 0, or -1 on invalid input, -2 when max_buckets is too small.
 * ------------------------------------------------------------------------- */
int oracle_plan(const int64_t* numels, const int32_t* tied_to, int32_t n_params,
                int32_t world, int64_t align, int64_t bucket_elems, int64_t* offsets,
                int64_t* info, int64_t* bucket_lo, int64_t* bucket_hi,
                int32_t max_buckets) {
  if (n_params < 0 || world < 1 || align < 1 || (n_params > 0 && (!numels || !offsets)) ||
      !info)
    return -1;
  std::vector<int32_t> owner(n_params);
  int64_t P = 0;
  for (int32_t i = 0; i < n_params; ++i) {
    if (numels[i] < 0) return -1;
    int32_t k = tied_to ? tied_to[i] : -1;
    if (k < 0) {
      owner[i] = i;
      offsets[i] = P;
      P += numels[i];
    } else {
      if (k >= i) return -1;
      owner[i] = owner[k];
      if (numels[owner[i]] != numels[i]) return -1;
      offsets[i] = offsets[owner[i]];
    }
  }
  int64_t Q = (int64_t)world * align;
  int64_t P_pad = (P + Q - 1) / Q * Q;
  int64_t S = P_pad / world;

  /* Buckets over the unique parameters, newest first. */
  std::vector<int64_t> lo, hi;
  if (bucket_elems <= 0) {
    lo.push_back(0);
    hi.push_back(P_pad);
  } else {
    int64_t cur_lo = -1, cur_hi = -1, cur_size = 0;
    for (int32_t i = n_params - 1; i >= 0; --i) {
      if (owner[i] != i) continue;
      int64_t n = numels[i];
      if (cur_size > 0 && cur_size + n > bucket_elems) {
        lo.push_back(cur_lo);
        hi.push_back(cur_hi);
        cur_size = 0;
      }
      if (cur_size == 0) {
        cur_hi = offsets[i] + n;
        cur_lo = offsets[i];
      } else {
        cur_lo = offsets[i];
      }
      cur_size += n;
    }
    if (cur_size > 0 || lo.empty()) {
      lo.push_back(cur_size > 0 ? cur_lo : 0);
      hi.push_back(cur_size > 0 ? cur_hi : 0);
    }
    /* The tail pad [P, P_pad) joins the bucket of the last-registered tensor,
     * which is the first bucket formed. */
    hi[0] = P_pad;
  }
  info[0] = P;
  info[1] = P_pad;
  info[2] = S;
  info[3] = (int64_t)lo.size();
  if ((int64_t)lo.size() > max_buckets) return -2;
  for (size_t b = 0; b < lo.size(); ++b) {
    if (bucket_lo) bucket_lo[b] = lo[b];
    if (bucket_hi) bucket_hi[b] = hi[b];
  }
  return 0;
}

/* Rank r's shard-local part of a flat range [flo, fhi): clamp to the shard and
 * shift to shard-local indices; may be empty (lo == hi). */
void oracle_shard_range(int64_t flo, int64_t fhi, int32_t rank, int64_t S, int64_t* lo,
                        int64_t* hi) {
  int64_t a = flo - (int64_t)rank * S, b = fhi - (int64_t)rank * S;
  *lo = a < 0 ? 0 : (a > S ? S : a);
  *hi = b < 0 ? 0 : (b > S ? S : b);
}

/* ---------------------------------------------------------------------------
 * O2. Persistent memory ledger, bytes per rank.
 * Bytes per parameter from the pages: DDP 2+2+(4+4+4) = 16 ([Dissection]
 * §1.1; [DP-to-ZeRO] "DDP 为什么单卡仍是 16P"); ZeRO-1 (2+2) + 12/dp
 * ([Dissection] §2.1); ZeRO-2 2 + (2+12)/dp ([Dissection] §2.2); ZeRO-3
 * (2+2+12)/dp ([Dissection] §2.3; [Lifecycle] persistent ledger).
 * stage: 0 = DDP, 1, 2, 3 = ZeRO stage. Returns the formula's bytes per
 * parameter as a double.
 * ------------------------------------------------------------------------- */
double oracle_ledger_bytes_per_param(int32_t stage, int32_t world) {
  double N = (double)world;
  switch (stage) {
    case 0: return 2.0 + 2.0 + (4.0 + 4.0 + 4.0);
    case 1: return (2.0 + 2.0) + 12.0 / N;
    case 2: return 2.0 + (2.0 + 12.0) / N;
    case 3: return (2.0 + 2.0 + 12.0) / N;
    default: return -1.0;
  }
}

/* The same ledger as the sum of the buffers a rank keeps for P_pad flat
 * elements (exact integers): bf16 params and bf16 grads are either the full
 * flat buffer (replicated) or one shard S = P_pad/N (sharded); the fp32
 * master, m and v are always one shard each once any stage shards them. */
int64_t oracle_ledger_kept_bytes(int32_t stage, int64_t P_pad, int32_t world) {
  int64_t S = P_pad / world;
  int64_t full_params = 2 * P_pad, full_grads = 2 * P_pad;
  switch (stage) {
    case 0: return full_params + full_grads + 4 * P_pad + 4 * P_pad + 4 * P_pad;
    case 1: return full_params + full_grads + (4 + 4 + 4) * S;
    case 2: return full_params + 2 * S + (4 + 4 + 4) * S;
    case 3: return 2 * S + 2 * S + (4 + 4 + 4) * S;
    default: return -1;
  }
}

/* The per-step fp32 scalars, for tests: out = {b1, b2, 1-b1, 1-b2, 1-b1^t,
 * 1-b2^t, lr, eps, 1-lr*wd, 1/N}. */
void oracle_adamw_scalars(double lr, double beta1, double beta2, double eps, double wd,
                          int64_t t, int32_t world, float* out) {
  Scalars s = make_scalars(lr, beta1, beta2, eps, wd, t, world);
  float v[10] = {s.b1, s.b2, s.omb1, s.omb2, s.bc1, s.bc2, s.lr, s.eps, s.decay, s.invN};
  std::memcpy(out, v, sizeof v);
}

/* ---------------------------------------------------------------------------
 * O3-O5. The shard-local step of rank `rank` on shard-local elements
 * [lo, hi) of a shard of S elements.
 *
 * O3 reduce: the N incoming slices are what a ReduceScatter delivers to this
 * rank: slice j is source rank j's local gradient restricted to this shard
 * ([Dissection] §2.1 Mechanism; [Lifecycle] "ReduceScatter: gradients
 * reduced, each rank keeps only its own shard"). The data-parallel gradient
 * is their mean ([DP-to-ZeRO] "Data Parallel 保证的数学语义": AllReduce to
 * the average gradient). Summed in fp32, j ascending, then times fp32(1/N).
 * O4 update: AdamW on this rank's master/m/v shard ([DP-to-ZeRO] "ZeRO Stage
 * 1": the owner rank updates its optimizer/parameter shard).
 * O5 cast + place: the updated master becomes the low-precision parameter in
 * this rank's slot of the flat buffer the AllGather fills ([DP-to-ZeRO]
 * "ZeRO Stage 1": all-gather updated parameter shards).
 *
 * grads[j] points at element 0 of slice j (S elements); master/m/v point at
 * element 0 of the shard; full_flat is the whole flat buffer [N*S] of the
 * parameter dtype, written at rank*S + i. Returns 0 or -1.
 * ------------------------------------------------------------------------- */
int oracle_shard_step(int32_t world, int32_t rank, int64_t S, int64_t lo, int64_t hi,
                      const void* const* grads, int32_t grad_dtype, float* master, float* m,
                      float* v, void* full_flat, int32_t param_dtype, double lr,
                      double beta1, double beta2, double eps, double wd, int64_t t) {
  if (world < 1 || rank < 0 || rank >= world || lo < 0 || hi < lo || hi > S || t < 1)
    return -1;
  if (!elem_bytes(param_dtype) || (grad_dtype != DT_BF16 && grad_dtype != DT_FP32))
    return -1;
  Scalars s = make_scalars(lr, beta1, beta2, eps, wd, t, world);
  int64_t slot = (int64_t)rank * S;
  for (int64_t i = lo; i < hi; ++i) {
    float acc = 0.0f;
    for (int32_t j = 0; j < world; ++j) acc = acc + load_grad(grads[j], grad_dtype, i);
    float g = acc * s.invN;
    adamw_element(s, g, master[i], m[i], v[i]);
    store_param(full_flat, param_dtype, slot + i, master[i]);
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Gradient clipping on the global norm, with the non-finite decision shared by
 * all ranks. [DP-to-ZeRO] "Gradient Accumulation 会改变生命周期" lists what a
 * sharded step must settle: whether clipping uses the global norm or the local
 * shard's, and whether overflow is decided by all ranks consistently; its
 * landing path (step 9) checks clipping by comparing single-step updates.
 * Readings: the global L2 norm of the reduced (mean) gradient over all P_pad
 * elements; each rank contributes the sum of squares of its shard and the N
 * partial sums are added in rank order (the emulated scalar AllReduce); the
 * coefficient is min(1, max_norm / (norm + 1e-6)) in double, rounded to fp32,
 * applied as g * coef after the mean; a non-finite norm (an Inf or NaN
 * anywhere) makes every rank skip the update, leaving master, m, v and the
 * parameter slot untouched.
 * ------------------------------------------------------------------------- */

/* Sum over i in [lo, hi), ascending, of g_i^2 in double, g_i being the step's
 * fp32 mean gradient (the square of an fp32 value is exact in double). */
double oracle_grad_sqnorm(int32_t world, int64_t S, int64_t lo, int64_t hi,
                          const void* const* grads, int32_t grad_dtype) {
  if (world < 1 || lo < 0 || hi < lo || hi > S) return -1.0;
  float invN = (float)(1.0 / (double)world);
  double sum = 0.0;
  for (int64_t i = lo; i < hi; ++i) {
    float acc = 0.0f;
    for (int32_t j = 0; j < world; ++j) acc = acc + load_grad(grads[j], grad_dtype, i);
    float g = acc * invN;
    sum = sum + (double)g * (double)g;
  }
  return sum;
}

/* The N ranks' partial sums of squares -> the clip coefficient and the shared
 * non-finite flag. */
void oracle_clip_coef(const double* rank_sqnorms, int32_t n, double max_norm, float* coef,
                      int32_t* nonfinite) {
  double total = 0.0;
  for (int32_t r = 0; r < n; ++r) total = total + rank_sqnorms[r];
  double norm = std::sqrt(total);
  *nonfinite = std::isfinite(norm) ? 0 : 1;
  double c = max_norm / (norm + 1e-6);
  *coef = *nonfinite ? 1.0f : (float)(c < 1.0 ? c : 1.0);
}

/* The shard step with the clip coefficient applied to the mean gradient and
 * the shared skip decision. */
int oracle_shard_step_clipped(int32_t world, int32_t rank, int64_t S, int64_t lo, int64_t hi,
                              const void* const* grads, int32_t grad_dtype, float* master,
                              float* m, float* v, void* full_flat, int32_t param_dtype,
                              double lr, double beta1, double beta2, double eps, double wd,
                              int64_t t, float coef, int32_t skip) {
  if (world < 1 || rank < 0 || rank >= world || lo < 0 || hi < lo || hi > S || t < 1)
    return -1;
  if (!elem_bytes(param_dtype) || (grad_dtype != DT_BF16 && grad_dtype != DT_FP32))
    return -1;
  if (skip) return 0;
  Scalars s = make_scalars(lr, beta1, beta2, eps, wd, t, world);
  int64_t slot = (int64_t)rank * S;
  for (int64_t i = lo; i < hi; ++i) {
    float acc = 0.0f;
    for (int32_t j = 0; j < world; ++j) acc = acc + load_grad(grads[j], grad_dtype, i);
    float g = (acc * s.invN) * coef;
    adamw_element(s, g, master[i], m[i], v[i]);
    store_param(full_flat, param_dtype, slot + i, master[i]);
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Gradient accumulation on the shard. [DP-to-ZeRO] "Gradient Accumulation 会
 * 改变生命周期": with G micro-batches per optimizer step one must decide whether
 * each micro-step ReduceScatters, whether to accumulate on the shard or on the
 * full tensor, and whether the loss is divided by G. Readings: every micro-step
 * ReduceScatters and its mean gradient is added into an fp32 accumulator of
 * this rank's shard (a_1 = 0 + mean_1, a_k = a_{k-1} + mean_k); the last
 * micro-step's slices go straight into the update with
 * g = (a_{G-1} + mean_G) * fp32(1/G), the average over the micro-batches.
 * ------------------------------------------------------------------------- */
int oracle_grad_accumulate(int32_t world, int64_t S, int64_t lo, int64_t hi,
                           const void* const* grads, int32_t grad_dtype, float* accum,
                           int32_t first) {
  if (world < 1 || lo < 0 || hi < lo || hi > S) return -1;
  float invN = (float)(1.0 / (double)world);
  for (int64_t i = lo; i < hi; ++i) {
    float acc = 0.0f;
    for (int32_t j = 0; j < world; ++j) acc = acc + load_grad(grads[j], grad_dtype, i);
    float mean = acc * invN;
    accum[i] = (first ? 0.0f : accum[i]) + mean;
  }
  return 0;
}

int oracle_shard_step_accumulated(int32_t world, int32_t rank, int64_t S, int64_t lo,
                                  int64_t hi, const void* const* grads, int32_t grad_dtype,
                                  const float* accum, int32_t micro_steps, float* master,
                                  float* m, float* v, void* full_flat, int32_t param_dtype,
                                  double lr, double beta1, double beta2, double eps, double wd,
                                  int64_t t) {
  if (world < 1 || rank < 0 || rank >= world || lo < 0 || hi < lo || hi > S || t < 1 ||
      micro_steps < 1)
    return -1;
  if (!elem_bytes(param_dtype) || (grad_dtype != DT_BF16 && grad_dtype != DT_FP32))
    return -1;
  Scalars s = make_scalars(lr, beta1, beta2, eps, wd, t, world);
  float invG = (float)(1.0 / (double)micro_steps);
  int64_t slot = (int64_t)rank * S;
  for (int64_t i = lo; i < hi; ++i) {
    float acc = 0.0f;
    for (int32_t j = 0; j < world; ++j) acc = acc + load_grad(grads[j], grad_dtype, i);
    float mean = acc * s.invN;
    float g = (accum[i] + mean) * invG;
    adamw_element(s, g, master[i], m[i], v[i]);
    store_param(full_flat, param_dtype, slot + i, master[i]);
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Clipping an accumulated gradient. The same section of [DP-to-ZeRO] asks both
 * questions at once: a job that accumulates G micro-batches and clips must
 * clip the gradient the update sees. Readings: that gradient is the micro-batch
 * average g = (a_{G-1} + mean_G) * fp32(1/G) of oracle_shard_step_accumulated;
 * its global norm is the sum over all shards of g^2 (each rank's part over its
 * shard, added in rank order by oracle_clip_coef, as for the plain step); the
 * update then sees g * coef, and a non-finite norm skips it on every rank.
 * ------------------------------------------------------------------------- */

/* Sum over i in [lo, hi), ascending, of g_i^2 in double, g_i the accumulated
 * step's fp32 gradient (the square of an fp32 value is exact in double). */
double oracle_grad_sqnorm_accumulated(int32_t world, int64_t S, int64_t lo, int64_t hi,
                                      const void* const* grads, int32_t grad_dtype,
                                      const float* accum, int32_t micro_steps) {
  if (world < 1 || lo < 0 || hi < lo || hi > S || micro_steps < 1) return -1.0;
  float invN = (float)(1.0 / (double)world);
  float invG = (float)(1.0 / (double)micro_steps);
  double sum = 0.0;
  for (int64_t i = lo; i < hi; ++i) {
    float acc = 0.0f;
    for (int32_t j = 0; j < world; ++j) acc = acc + load_grad(grads[j], grad_dtype, i);
    float mean = acc * invN;
    float g = (accum[i] + mean) * invG;
    sum = sum + (double)g * (double)g;
  }
  return sum;
}

/* The accumulated step with the clip coefficient and the shared skip. */
int oracle_shard_step_accumulated_clipped(int32_t world, int32_t rank, int64_t S, int64_t lo,
                                          int64_t hi, const void* const* grads,
                                          int32_t grad_dtype, const float* accum,
                                          int32_t micro_steps, float* master, float* m,
                                          float* v, void* full_flat, int32_t param_dtype,
                                          double lr, double beta1, double beta2, double eps,
                                          double wd, int64_t t, float coef, int32_t skip) {
  if (world < 1 || rank < 0 || rank >= world || lo < 0 || hi < lo || hi > S || t < 1 ||
      micro_steps < 1)
    return -1;
  if (!elem_bytes(param_dtype) || (grad_dtype != DT_BF16 && grad_dtype != DT_FP32))
    return -1;
  if (skip) return 0;
  Scalars s = make_scalars(lr, beta1, beta2, eps, wd, t, world);
  float invG = (float)(1.0 / (double)micro_steps);
  int64_t slot = (int64_t)rank * S;
  for (int64_t i = lo; i < hi; ++i) {
    float acc = 0.0f;
    for (int32_t j = 0; j < world; ++j) acc = acc + load_grad(grads[j], grad_dtype, i);
    float mean = acc * s.invN;
    float g = ((accum[i] + mean) * invG) * coef;
    adamw_element(s, g, master[i], m[i], v[i]);
    store_param(full_flat, param_dtype, slot + i, master[i]);
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Per-parameter row sharding (FSDP2) and the gather side of a wrap unit.
 * [DP-to-ZeRO] "ZeRO 与 FSDP 的关系": FSDP2 keeps per-parameter sharded state;
 * [Lifecycle] "The parameter lifecycle, one module at a time": AllGather the
 * module's parameters before its compute, reshard after (to 1/N, or, with an
 * integer reshard_after_forward, to a smaller world); [Dissection] §7: a
 * 768-element layer norm over 64 ranks gives 12-element shards.
 * Readings: each parameter is cut along dim 0 into chunks of c = ceil(dim0/N)
 * rows, rank r holding rows [r*c, min((r+1)*c, dim0)) (none when r*c >= dim0),
 * padded with zero rows to c; a rank's local buffer is its padded chunks back
 * to back in registration order (tied parameters once), padded with zeros to a
 * multiple of align; the AllGather output is the N local buffers rank-major.
 * ------------------------------------------------------------------------- */
int oracle_rows_plan(const int64_t* dim0, const int64_t* numels, const int32_t* tied_to,
                     int32_t n_params, int32_t world, int64_t align, int64_t* offsets,
                     int64_t* rows_per_rank, int64_t* row_elems, int64_t* S_out) {
  if (world < 1 || align < 1 || n_params < 0) return -1;
  int64_t local = 0;
  for (int32_t i = 0; i < n_params; ++i) {
    if (numels[i] < 0 || dim0[i] < 0 || (dim0[i] == 0 && numels[i] != 0) ||
        (dim0[i] > 0 && numels[i] % dim0[i] != 0))
      return -1;
    int32_t k = tied_to ? tied_to[i] : -1;
    if (k >= 0) {
      if (k >= i) return -1;
      offsets[i] = offsets[k];
      rows_per_rank[i] = rows_per_rank[k];
      row_elems[i] = row_elems[k];
      continue;
    }
    row_elems[i] = dim0[i] > 0 ? numels[i] / dim0[i] : 0;
    rows_per_rank[i] = (dim0[i] + world - 1) / world;
    offsets[i] = local;
    local += rows_per_rank[i] * row_elems[i];
  }
  *S_out = (local + align - 1) / align * align;
  return 0;
}

/* Rows of parameter i that rank r holds. */
static int64_t rows_held(int64_t dim0, int64_t c, int32_t r) {
  int64_t first = (int64_t)r * c;
  if (first >= dim0) return 0;
  return first + c <= dim0 ? c : dim0 - first;
}

/* The copy-out: gathered [N][S] -> each owner parameter's full tensor. */
void oracle_unshard(const int64_t* dim0, const int64_t* offsets, const int64_t* rows_per_rank,
                    const int64_t* row_elems, const int32_t* tied_to, int32_t n_params,
                    int32_t world, int64_t S, int32_t elem_size, const void* gathered,
                    void* const* params) {
  for (int32_t i = 0; i < n_params; ++i) {
    if (tied_to && tied_to[i] >= 0) continue;
    int64_t row_bytes = row_elems[i] * elem_size;
    for (int32_t r = 0; r < world; ++r) {
      int64_t rows = rows_held(dim0[i], rows_per_rank[i], r);
      const uint8_t* src = static_cast<const uint8_t*>(gathered) +
                           ((size_t)r * S + offsets[i]) * elem_size;
      uint8_t* dst = static_cast<uint8_t*>(params[i]) + (size_t)r * rows_per_rank[i] * row_bytes;
      std::memcpy(dst, src, (size_t)(rows * row_bytes));
    }
  }
}

/* The copy-in / reshard: rank r's local buffer from the full parameters. */
void oracle_shard_rows(const int64_t* dim0, const int64_t* offsets, const int64_t* rows_per_rank,
                       const int64_t* row_elems, const int32_t* tied_to, int32_t n_params,
                       int32_t rank, int64_t S, int32_t elem_size, const void* const* params,
                       void* local) {
  std::memset(local, 0, (size_t)S * elem_size);
  for (int32_t i = 0; i < n_params; ++i) {
    if (tied_to && tied_to[i] >= 0) continue;
    int64_t row_bytes = row_elems[i] * elem_size;
    int64_t rows = rows_held(dim0[i], rows_per_rank[i], rank);
    const uint8_t* src = static_cast<const uint8_t*>(params[i]) +
                         (size_t)rank * rows_per_rank[i] * row_bytes;
    uint8_t* dst = static_cast<uint8_t*>(local) + (size_t)offsets[i] * elem_size;
    std::memcpy(dst, src, (size_t)(rows * row_bytes));
  }
}

/* ---------------------------------------------------------------------------
 * O7. The unsharded data-parallel step every DDP replica runs ([DP-to-ZeRO]
 * "DDP 为什么单卡仍是 16P" and "Data Parallel 保证的数学语义"): AllReduce the
 * N local gradients to their mean over the whole flat buffer, run AdamW on
 * the full fp32 master/m/v, cast the full parameter buffer. ZeRO-1 only
 * restructures this AllReduce ([Dissection] §2.1 Communication cost), so the
 * concatenation of the N shard-local steps must reproduce it exactly.
 * local_grads[j] points at source rank j's full local gradient [P_pad].
 * ------------------------------------------------------------------------- */
int oracle_ddp_step(int32_t world, int64_t P_pad, const void* const* local_grads,
                    int32_t grad_dtype, float* master, float* m, float* v, void* params,
                    int32_t param_dtype, double lr, double beta1, double beta2, double eps,
                    double wd, int64_t t) {
  if (world < 1 || P_pad < 0 || t < 1 || !elem_bytes(param_dtype)) return -1;
  Scalars s = make_scalars(lr, beta1, beta2, eps, wd, t, world);
  /* AllReduce (mean). */
  std::vector<float> mean(P_pad);
  for (int64_t i = 0; i < P_pad; ++i) {
    float acc = 0.0f;
    for (int32_t j = 0; j < world; ++j) acc = acc + load_grad(local_grads[j], grad_dtype, i);
    mean[i] = acc * s.invN;
  }
  /* Full optimizer step on the replica. */
  for (int64_t i = 0; i < P_pad; ++i) adamw_element(s, mean[i], master[i], m[i], v[i]);
  /* Full low-precision parameters. */
  for (int64_t i = 0; i < P_pad; ++i) store_param(params, param_dtype, i, master[i]);
  return 0;
}

/* ---------------------------------------------------------------------------
 * O6. AllGather emulation: slot j of the flat buffer receives shard j
 * ([DP-to-ZeRO] "ZeRO Stage 1": all-gather updated parameter shards, all ranks
 * again hold identical full parameters). A NULL source leaves its slot as is.
 * ------------------------------------------------------------------------- */
void oracle_gather(int32_t world, int64_t S, int32_t elem_size, const void* const* shards,
                   void* full_flat) {
  for (int32_t j = 0; j < world; ++j) {
    if (!shards[j]) continue;
    std::memcpy(static_cast<uint8_t*>(full_flat) + (size_t)j * S * elem_size, shards[j],
                (size_t)S * elem_size);
  }
}

/* Casts, exposed for tests. */
uint16_t oracle_bf16_rne(float x) { return (uint16_t)round_keep_high(x, 16); }
uint32_t oracle_fp24_rne(float x) { return round_keep_high(x, 8); }
void oracle_bf16_rne_array(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint16_t)round_keep_high(x[i], 16);
}
void oracle_bf16_rne_bits_range(uint32_t first, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = (uint16_t)round_keep_high(bits_float(first + (uint32_t)i), 16);
}
/* The 3-byte cast of the fp32 patterns first, first + 1, ... (mod 2^32),
 * stored as the parameter slot stores it: 3 bytes per value, little-endian. */
void oracle_fp24_rne_bits_range(uint32_t first, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    uint32_t q = round_keep_high(bits_float(first + (uint32_t)i), 8);
    out[3 * i] = (uint8_t)(q & 0xFFu);
    out[3 * i + 1] = (uint8_t)((q >> 8) & 0xFFu);
    out[3 * i + 2] = (uint8_t)((q >> 16) & 0xFFu);
  }
}

}  // extern "C"
