// plan.cpp — the flat-parameter planner (zs_flatten_plan and its queries).
//
// Layout ("ZeRO vs FSDP: A Rigorous Dissection", §3.2 The FlatParameter
// Abstraction; "从 Data Parallel 到 ZeRO/FSDP", "ZeRO Stage 1", "Shared
// Parameters 与 Tied Weights", "ReduceScatter 必须尽早释放 Gradient"):
// unique parameters are packed back to back in registration order, a tied
// parameter reuses its owner's storage, the total is padded to a multiple of
// world*align so that N equal contiguous shards exist, and buckets of whole
// tensors are formed newest-first (backward readiness order).
#include <mutex>
#include <new>
#include <unordered_set>

#include "zs_internal.h"

namespace {

std::mutex g_live_mu;
std::unordered_set<const zs_plan*>& live_plans() {
  static std::unordered_set<const zs_plan*> s;
  return s;
}

bool add_overflows(int64_t a, int64_t b) { return b > 0 && a > INT64_MAX - b; }

}  // namespace

namespace zs {
bool plan_is_live(const zs_plan* plan) {
  if (!plan) return false;
  std::lock_guard<std::mutex> lock(g_live_mu);
  return live_plans().count(plan) != 0 && plan->magic == kPlanMagic;
}
}  // namespace zs

extern "C" zs_status zs_flatten_plan(const int64_t* numels, const int32_t* tied_to,
                                     int32_t n_params, int32_t world, int64_t align_elems,
                                     int64_t bucket_elems, zs_plan** out) {
  zs::clear_error();
  if (!out) return zs::fail(ZS_ERR_INVAL, "zs_flatten_plan: out is NULL");
  *out = nullptr;
  if (n_params < 0) return zs::fail(ZS_ERR_INVAL, "zs_flatten_plan: n_params < 0");
  if (n_params > 0 && !numels) return zs::fail(ZS_ERR_INVAL, "zs_flatten_plan: numels is NULL");
  if (world < 1 || world > ZS_MAX_WORLD)
    return zs::fail(ZS_ERR_RANGE, "zs_flatten_plan: world %d outside 1..%d", world,
                    ZS_MAX_WORLD);
  if (align_elems < 1 || align_elems > (int64_t(1) << 32))
    return zs::fail(ZS_ERR_RANGE, "zs_flatten_plan: align_elems %lld out of range",
                    (long long)align_elems);
  if (bucket_elems < 0) return zs::fail(ZS_ERR_RANGE, "zs_flatten_plan: bucket_elems < 0");

  zs_plan* p = new (std::nothrow) zs_plan();
  if (!p) return zs::fail(ZS_ERR_NOMEM, "zs_flatten_plan: out of host memory");
  try {
    p->numels.assign(numels, numels + n_params);
    p->offsets.assign(n_params, 0);
    p->owner.assign(n_params, 0);
  } catch (...) {
    delete p;
    return zs::fail(ZS_ERR_NOMEM, "zs_flatten_plan: out of host memory");
  }
  p->layout = zs::kLayoutFlat;
  p->world = world;
  p->n_params = n_params;
  p->align = align_elems;
  p->bucket_elems = bucket_elems;

  int64_t total = 0;
  for (int32_t i = 0; i < n_params; ++i) {
    int64_t n = numels[i];
    if (n < 0) {
      delete p;
      return zs::fail(ZS_ERR_INVAL, "zs_flatten_plan: numels[%d] < 0", i);
    }
    int32_t t = tied_to ? tied_to[i] : -1;
    if (t < 0) {
      if (add_overflows(total, n)) {
        delete p;
        return zs::fail(ZS_ERR_RANGE, "zs_flatten_plan: total size overflows int64");
      }
      p->owner[i] = i;
      p->offsets[i] = total;
      total += n;
      continue;
    }
    if (t >= i) {
      delete p;
      return zs::fail(ZS_ERR_INVAL, "zs_flatten_plan: tied_to[%d] = %d is not an earlier param",
                      i, t);
    }
    int32_t root = p->owner[t];
    if (numels[root] != n) {
      delete p;
      return zs::fail(ZS_ERR_INVAL, "zs_flatten_plan: tied param %d has %lld elements, owner %d has %lld",
                      i, (long long)n, root, (long long)numels[root]);
    }
    p->owner[i] = root;
    p->offsets[i] = p->offsets[root];
  }
  const int64_t quantum = (int64_t)world * align_elems;
  if (add_overflows(total, quantum - 1)) {
    delete p;
    return zs::fail(ZS_ERR_RANGE, "zs_flatten_plan: padded size overflows int64");
  }
  p->P = total;
  p->P_pad = (total + quantum - 1) / quantum * quantum;
  p->S = p->P_pad / world;

  // Buckets, first ready first: walk the owners from the last registered.
  try {
    if (bucket_elems == 0) {
      p->bucket_lo.push_back(0);
      p->bucket_hi.push_back(p->P_pad);
    } else {
      int64_t size = 0, lo = 0, hi = 0;
      for (int32_t i = n_params - 1; i >= 0; --i) {
        if (p->owner[i] != i) continue;
        const int64_t n = p->numels[i];
        if (size > 0 && size + n > bucket_elems) {
          p->bucket_lo.push_back(lo);
          p->bucket_hi.push_back(hi);
          size = 0;
        }
        if (size == 0) hi = p->offsets[i] + n;
        lo = p->offsets[i];
        size += n;
      }
      if (size > 0 || p->bucket_lo.empty()) {
        p->bucket_lo.push_back(size > 0 ? lo : 0);
        p->bucket_hi.push_back(size > 0 ? hi : 0);
      }
      p->bucket_hi[0] = p->P_pad;  // the tail pad rides with the first bucket
    }
  } catch (...) {
    delete p;
    return zs::fail(ZS_ERR_NOMEM, "zs_flatten_plan: out of host memory");
  }
  p->magic = zs::kPlanMagic;
  {
    std::lock_guard<std::mutex> lock(g_live_mu);
    live_plans().insert(p);
  }
  *out = p;
  return ZS_OK;
}

extern "C" zs_status zs_plan_info(const zs_plan* plan, int64_t* P, int64_t* P_pad, int64_t* S,
                                  int32_t* n_buckets, int32_t* world, int32_t* n_params) {
  zs::clear_error();
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "zs_plan_info: not a live plan");
  if (P) *P = plan->P;
  if (P_pad) *P_pad = plan->P_pad;
  if (S) *S = plan->S;
  if (n_buckets) *n_buckets = (int32_t)plan->bucket_lo.size();
  if (world) *world = plan->world;
  if (n_params) *n_params = plan->n_params;
  return ZS_OK;
}

extern "C" zs_status zs_plan_offsets(const zs_plan* plan, int64_t* offsets, int32_t n_params) {
  zs::clear_error();
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "zs_plan_offsets: not a live plan");
  if (n_params != plan->n_params)
    return zs::fail(ZS_ERR_RANGE, "zs_plan_offsets: plan has %d params, caller passed %d",
                    plan->n_params, n_params);
  if (n_params > 0 && !offsets) return zs::fail(ZS_ERR_INVAL, "zs_plan_offsets: offsets is NULL");
  for (int32_t i = 0; i < n_params; ++i) offsets[i] = plan->offsets[i];
  return ZS_OK;
}

extern "C" zs_status zs_plan_bucket_range(const zs_plan* plan, int32_t bucket, int64_t* flat_lo,
                                          int64_t* flat_hi) {
  zs::clear_error();
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "zs_plan_bucket_range: not a live plan");
  if (bucket < 0 || bucket >= (int32_t)plan->bucket_lo.size())
    return zs::fail(ZS_ERR_RANGE, "zs_plan_bucket_range: bucket %d out of range", bucket);
  if (flat_lo) *flat_lo = plan->bucket_lo[bucket];
  if (flat_hi) *flat_hi = plan->bucket_hi[bucket];
  return ZS_OK;
}

extern "C" zs_status zs_plan_bucket(const zs_plan* plan, int32_t bucket, int32_t rank,
                                    int64_t* lo, int64_t* hi) {
  zs::clear_error();
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "zs_plan_bucket: not a live plan");
  if (bucket < 0 || bucket >= (int32_t)plan->bucket_lo.size())
    return zs::fail(ZS_ERR_RANGE, "zs_plan_bucket: bucket %d out of range", bucket);
  if (rank < 0 || rank >= plan->world)
    return zs::fail(ZS_ERR_RANGE, "zs_plan_bucket: rank %d out of range", rank);
  const int64_t base = (int64_t)rank * plan->S;
  auto clamp = [&](int64_t x) {
    int64_t y = x - base;
    return y < 0 ? int64_t(0) : (y > plan->S ? plan->S : y);
  };
  if (lo) *lo = clamp(plan->bucket_lo[bucket]);
  if (hi) *hi = clamp(plan->bucket_hi[bucket]);
  return ZS_OK;
}

extern "C" zs_status zs_plan_free(zs_plan* plan) {
  zs::clear_error();
  {
    std::lock_guard<std::mutex> lock(g_live_mu);
    auto it = live_plans().find(plan);
    if (!plan || it == live_plans().end())
      return zs::fail(ZS_ERR_INVAL, "zs_plan_free: not a live plan (freed twice?)");
    live_plans().erase(it);
  }
  plan->magic = 0;
  delete plan;
  return ZS_OK;
}

// The per-parameter row layout of FSDP2 ("从 Data Parallel 到 ZeRO/FSDP", "ZeRO 与
// FSDP 的关系": fully_shard keeps per-parameter sharded state): parameter i is
// cut along dim 0 into N chunks of c_i = ceil(dim0_i / N) rows; rank r holds
// rows [r*c_i, min((r+1)*c_i, dim0_i)) (possibly none), padded to c_i rows.
// A rank's local buffer is its padded chunks back to back in registration
// order (tied parameters once), padded at the end to a multiple of
// align_elems: S = that length. The AllGather of the N local buffers is the
// rank-major [N][S] buffer that zs_unshard copies out into parameters.
extern "C" zs_status zs_rows_plan(const int64_t* dim0, const int64_t* numels,
                                  const int32_t* tied_to, int32_t n_params, int32_t world,
                                  int64_t align_elems, zs_plan** out) {
  zs::clear_error();
  if (!out) return zs::fail(ZS_ERR_INVAL, "zs_rows_plan: out is NULL");
  *out = nullptr;
  if (n_params < 0) return zs::fail(ZS_ERR_INVAL, "zs_rows_plan: n_params < 0");
  if (n_params > 0 && (!numels || !dim0))
    return zs::fail(ZS_ERR_INVAL, "zs_rows_plan: numels or dim0 is NULL");
  if (world < 1 || world > ZS_MAX_WORLD)
    return zs::fail(ZS_ERR_RANGE, "zs_rows_plan: world %d outside 1..%d", world, ZS_MAX_WORLD);
  if (align_elems < 1 || align_elems > (int64_t(1) << 32))
    return zs::fail(ZS_ERR_RANGE, "zs_rows_plan: align_elems %lld out of range",
                    (long long)align_elems);
  zs_plan* p = new (std::nothrow) zs_plan();
  if (!p) return zs::fail(ZS_ERR_NOMEM, "zs_rows_plan: out of host memory");
  try {
    p->numels.assign(numels, numels + n_params);
    p->dim0.assign(dim0, dim0 + n_params);
    p->offsets.assign(n_params, 0);
    p->owner.assign(n_params, 0);
    p->row_elems.assign(n_params, 0);
    p->rows_per_rank.assign(n_params, 0);
  } catch (...) {
    delete p;
    return zs::fail(ZS_ERR_NOMEM, "zs_rows_plan: out of host memory");
  }
  p->layout = zs::kLayoutRows;
  p->world = world;
  p->n_params = n_params;
  p->align = align_elems;
  p->bucket_elems = 0;
  int64_t local = 0, total = 0;
  for (int32_t i = 0; i < n_params; ++i) {
    const int64_t n = numels[i], d = dim0[i];
    if (n < 0 || d < 0 || (d == 0 && n != 0) || (d > 0 && n % d != 0)) {
      delete p;
      return zs::fail(ZS_ERR_INVAL, "zs_rows_plan: param %d has %lld elements in %lld rows", i,
                      (long long)n, (long long)d);
    }
    const int32_t t = tied_to ? tied_to[i] : -1;
    if (t >= 0) {
      if (t >= i) {
        delete p;
        return zs::fail(ZS_ERR_INVAL, "zs_rows_plan: tied_to[%d] = %d is not an earlier param", i, t);
      }
      const int32_t root = p->owner[t];
      if (numels[root] != n || dim0[root] != d) {
        delete p;
        return zs::fail(ZS_ERR_INVAL, "zs_rows_plan: tied param %d differs from its owner %d", i, root);
      }
      p->owner[i] = root;
      p->offsets[i] = p->offsets[root];
      p->row_elems[i] = p->row_elems[root];
      p->rows_per_rank[i] = p->rows_per_rank[root];
      continue;
    }
    p->owner[i] = i;
    p->row_elems[i] = d > 0 ? n / d : 0;
    p->rows_per_rank[i] = (d + world - 1) / world;
    const int64_t seg = p->rows_per_rank[i] * p->row_elems[i];
    if (add_overflows(local, seg) || add_overflows(total, n)) {
      delete p;
      return zs::fail(ZS_ERR_RANGE, "zs_rows_plan: sizes overflow int64");
    }
    p->offsets[i] = local;
    local += seg;
    total += n;
  }
  if (add_overflows(local, align_elems - 1)) {
    delete p;
    return zs::fail(ZS_ERR_RANGE, "zs_rows_plan: padded size overflows int64");
  }
  p->S = (local + align_elems - 1) / align_elems * align_elems;
  p->P = total;
  p->P_pad = p->S * world;
  try {
    p->bucket_lo.push_back(0);
    p->bucket_hi.push_back(p->P_pad);
  } catch (...) {
    delete p;
    return zs::fail(ZS_ERR_NOMEM, "zs_rows_plan: out of host memory");
  }
  p->magic = zs::kPlanMagic;
  {
    std::lock_guard<std::mutex> lock(g_live_mu);
    live_plans().insert(p);
  }
  *out = p;
  return ZS_OK;
}

extern "C" zs_status zs_plan_rows(const zs_plan* plan, int64_t* rows_per_rank,
                                  int64_t* row_elems, int32_t n_params) {
  zs::clear_error();
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "zs_plan_rows: not a live plan");
  if (plan->layout != zs::kLayoutRows)
    return zs::fail(ZS_ERR_UNSUPPORTED, "zs_plan_rows: not a row-sharded plan");
  if (n_params != plan->n_params)
    return zs::fail(ZS_ERR_RANGE, "zs_plan_rows: plan has %d params, caller passed %d",
                    plan->n_params, n_params);
  for (int32_t i = 0; i < n_params; ++i) {
    if (rows_per_rank) rows_per_rank[i] = plan->rows_per_rank[i];
    if (row_elems) row_elems[i] = plan->row_elems[i];
  }
  return ZS_OK;
}
