// trace.cpp — the per-call trace, finding where ranks' traces diverge, and the
// NVTX range around each traced call.
//
// "从 Data Parallel 到 ZeRO/FSDP", "训练 Hang 应按 Collective 顺序排查": ZeRO/FSDP
// insert collectives from hooks, so ranks that enter modules in a different
// order or number of times wait in different collectives (one in a parameter
// AllGather, another already in a gradient ReduceScatter); to find the first
// point where the ranks' programs part, record for every collective its
// sequence number, process group, tensor numel, dtype, module and phase.
//
// Every call of this library that stands at a collective of the real system
// (the step after the ReduceScatter, the accumulation, the norm and its scalar
// AllReduce, the AllGather's assembly and copy-out, the checkpoint) appends
// one line to the trace when tracing is on:
//   seq=<n> call=<name> plan=<id> world=<N> S=<shard elements> rank=<r>
//   lo=<lo> hi=<hi> grad=<dtype> param=<dtype> step=<t> status=<code>
// plan is a hash of the plan's parameter list and layout (the same on every
// rank of one model; the "module" of the passage), world the group size.
// Tracing is off unless ZS_TRACE names a file (read at the first traced
// call) or zs_set_trace is called; in the path, %r becomes the RANK
// environment variable (0 if unset) and %p the process id.
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <cinttypes>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "zs_internal.h"

namespace {

std::mutex g_trace_mu;
FILE* g_trace_file = nullptr;     // guarded by g_trace_mu
std::atomic<bool> g_trace_env_read{false};  // set under g_trace_mu
std::atomic<bool> g_trace_on{false};
std::atomic<uint64_t> g_trace_seq{0};

std::string expand_path(const char* path) {
  std::string out;
  const char* rank = std::getenv("RANK");
  for (const char* p = path; *p; ++p) {
    if (p[0] == '%' && p[1] == 'r') {
      out += rank && *rank ? rank : "0";
      ++p;
    } else if (p[0] == '%' && p[1] == 'p') {
      out += std::to_string((long long)getpid());
      ++p;
    } else {
      out += *p;
    }
  }
  return out;
}

// Opens (appending) the trace file, or turns tracing off for NULL. Caller
// holds g_trace_mu.
bool open_trace_locked(const char* path) {
  if (g_trace_file) {
    std::fclose(g_trace_file);
    g_trace_file = nullptr;
  }
  g_trace_on.store(false);
  if (!path || !*path) return true;
  g_trace_file = std::fopen(expand_path(path).c_str(), "a");
  if (!g_trace_file) return false;
  g_trace_seq.store(0);
  g_trace_on.store(true);
  return true;
}

// FNV-1a over the plan's parameter list and layout.
uint64_t plan_id(const zs_plan* p) {
  uint64_t h = 1469598103934665603ull;
  auto mix = [&h](const void* data, size_t n) {
    const unsigned char* b = static_cast<const unsigned char*>(data);
    for (size_t i = 0; i < n; ++i) h = (h ^ b[i]) * 1099511628211ull;
  };
  mix(&p->layout, sizeof p->layout);
  mix(&p->world, sizeof p->world);
  mix(&p->n_params, sizeof p->n_params);
  mix(&p->align, sizeof p->align);
  mix(&p->bucket_elems, sizeof p->bucket_elems);
  if (!p->numels.empty()) mix(p->numels.data(), p->numels.size() * sizeof(int64_t));
  if (!p->owner.empty()) mix(p->owner.data(), p->owner.size() * sizeof(int32_t));
  if (!p->dim0.empty()) mix(p->dim0.data(), p->dim0.size() * sizeof(int64_t));
  return h;
}

const char* dtype_name(int dt) {
  switch (dt) {
    case ZS_BF16: return "bf16";
    case ZS_FP32: return "fp32";
    case ZS_FP24: return "fp24";
    default: return "-";
  }
}

// The fields two ranks must agree on at the same sequence number.
const char* const kSignatureKeys[] = {"call", "plan", "world", "S", "grad", "param", "step"};

struct Record {
  std::map<std::string, std::string> kv;
  std::string line;
};

bool read_trace(const char* path, std::vector<Record>* out) {
  FILE* f = std::fopen(path, "r");
  if (!f) return false;
  char buf[1024];
  while (std::fgets(buf, sizeof buf, f)) {
    Record r;
    r.line = buf;
    while (!r.line.empty() && (r.line.back() == '\n' || r.line.back() == '\r')) r.line.pop_back();
    size_t i = 0;
    while (i < r.line.size()) {
      while (i < r.line.size() && r.line[i] == ' ') ++i;
      const size_t j = r.line.find(' ', i);
      const std::string tok = r.line.substr(i, j == std::string::npos ? std::string::npos : j - i);
      const size_t eq = tok.find('=');
      if (eq != std::string::npos) r.kv[tok.substr(0, eq)] = tok.substr(eq + 1);
      if (j == std::string::npos) break;
      i = j + 1;
    }
    if (!r.kv.empty()) out->push_back(std::move(r));
  }
  std::fclose(f);
  return true;
}

std::string signature(const Record& r) {
  std::string s;
  for (const char* k : kSignatureKeys) {
    auto it = r.kv.find(k);
    s += k;
    s += '=';
    s += it == r.kv.end() ? "?" : it->second;
    s += ' ';
  }
  return s;
}

}  // namespace

namespace zs {

CallRange::CallRange(const char* name) { nvtxRangePushA(name); }
CallRange::~CallRange() { nvtxRangePop(); }

zs_status traced(zs_status st, const char* call, const zs_plan* plan, int32_t rank, int64_t lo,
                 int64_t hi, int grad_dtype, int param_dtype, int64_t step, int32_t world) {
  if (!g_trace_on.load(std::memory_order_relaxed)) {
    // Off: one atomic load per call once ZS_TRACE has been looked at.
    if (g_trace_env_read.load(std::memory_order_acquire)) return st;
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (g_trace_env_read.load()) return st;
    g_trace_env_read.store(true, std::memory_order_release);
    if (const char* env = std::getenv("ZS_TRACE")) open_trace_locked(env);
    if (!g_trace_on.load()) return st;
  }
  const bool live = plan_is_live(plan);
  char id[24];
  if (live) std::snprintf(id, sizeof id, "%016" PRIx64, plan_id(plan));
  else std::snprintf(id, sizeof id, "-");
  const uint64_t seq = g_trace_seq.fetch_add(1);
  char line[512];
  std::snprintf(line, sizeof line,
                "seq=%" PRIu64 " call=%s plan=%s world=%d S=%lld rank=%d lo=%lld hi=%lld "
                "grad=%s param=%s step=%lld status=%d\n",
                seq, call, id, live ? plan->world : world, live ? (long long)plan->S : -1LL,
                rank, (long long)lo, (long long)hi, dtype_name(grad_dtype),
                dtype_name(param_dtype), (long long)step, (int)st);
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (g_trace_file) {
    std::fputs(line, g_trace_file);
    std::fflush(g_trace_file);
  }
  return st;
}

}  // namespace zs

extern "C" zs_status zs_set_trace(const char* path) {
  zs::clear_error();
  std::lock_guard<std::mutex> lock(g_trace_mu);
  g_trace_env_read.store(true);  // an explicit setting wins over ZS_TRACE
  if (!open_trace_locked(path))
    return zs::fail(ZS_ERR_IO, "zs_set_trace: cannot open %s", path);
  return ZS_OK;
}

extern "C" zs_status zs_trace_first_divergence(const char* const* paths, int32_t n_paths,
                                               int64_t* seq_out, char* detail,
                                               int64_t detail_bytes) {
  static const char* fn = "zs_trace_first_divergence";
  zs::clear_error();
  if (!paths || n_paths < 2 || !seq_out)
    return zs::fail(ZS_ERR_INVAL, "%s: need two or more trace paths and seq_out", fn);
  std::vector<std::vector<Record>> traces(n_paths);
  for (int32_t k = 0; k < n_paths; ++k) {
    if (!paths[k]) return zs::fail(ZS_ERR_INVAL, "%s: paths[%d] is NULL", fn, k);
    try {
      if (!read_trace(paths[k], &traces[k]))
        return zs::fail(ZS_ERR_IO, "%s: cannot read %s", fn, paths[k]);
    } catch (...) {
      return zs::fail(ZS_ERR_NOMEM, "%s: out of host memory", fn);
    }
  }
  size_t longest = 0;
  for (const auto& t : traces) longest = std::max(longest, t.size());
  std::string msg;
  int64_t at = -1;
  for (size_t i = 0; i < longest && at < 0; ++i) {
    // The first trace holding record i fixes the signature the others must match.
    std::string ref;
    bool have_ref = false, differ = false;
    for (const auto& t : traces) {
      if (i >= t.size()) {
        differ = true;
        continue;
      }
      const std::string sig = signature(t[i]);
      if (!have_ref) {
        ref = sig;
        have_ref = true;
      } else if (sig != ref) {
        differ = true;
      }
    }
    if (!differ) continue;
    at = (int64_t)i;
    msg = "record " + std::to_string(i) + ":";
    for (int32_t k = 0; k < n_paths; ++k) {
      msg += k == 0 ? " " : " | ";
      msg += paths[k];
      msg += ": ";
      msg += i < traces[k].size() ? traces[k][i].line
                                  : "ends after " + std::to_string(traces[k].size()) + " records";
    }
  }
  *seq_out = at;
  if (detail && detail_bytes > 0) {
    std::snprintf(detail, (size_t)detail_bytes, "%s", at < 0 ? "" : msg.c_str());
  }
  return ZS_OK;
}
