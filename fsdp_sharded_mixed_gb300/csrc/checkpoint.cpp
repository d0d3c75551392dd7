// checkpoint.cpp — sharded checkpoint of the optimizer state, and restore into
// another world size or layout.
//
// "从 Data Parallel 到 ZeRO/FSDP", "Checkpoint 不能假设每个 Rank 都有完整模型":
// under ZeRO-3/FSDP no rank holds the whole model, so each rank writes its own
// shards and the metadata that places them in the global tensors; restoring
// into another world size means resharding; a consistent checkpoint carries
// the master weights and moments, the global step and the sharding metadata,
// and a restore counts only if the next update equals the uninterrupted run's.
// Its landing path (step 10) asks for saving, fault injection, and restores at
// the same and at another world size.
//
// File of one rank (little-endian; every offset below is in the header):
//   Header (128 bytes), then the parameter list and the layout (numels,
//   offsets, rows per rank, row length as int64[n], then ties as int32[n]),
//   then, each at a 4 KiB boundary, the three fp32 arrays of S elements
//   (master, exp_avg, exp_avg_sq), then per array one 64-bit checksum per
//   block (block_hash.h) of block_bytes.
// Element e of parameter i is a place in the global tensor whatever the
// layout, so a load maps every element of the new rank's shard to (old rank,
// old local index) through the two layouts (flat: global flat index; rows:
// rank = e / (rows per rank * row length)), reads only the blocks it needs,
// and checks every block it reads: on the device, where the block landed in
// HBM, when the block lies whole inside one copy; on the host, before the
// copy, otherwise (the edge blocks of a reshard, and host-resident state).
// Padding elements of the new shard are zero, as the initial state's are.
//
// No call here allocates device memory: device-resident state moves through
// pinned host staging, so a restore cannot fail for want of HBM next to a
// model that fills it.
#include <cuda_runtime.h>
#include <errno.h>
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <condition_variable>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "block_hash.h"
#include "zs_internal.h"

#if !defined(__BYTE_ORDER__) || __BYTE_ORDER__ != __ORDER_LITTLE_ENDIAN__
#error "the checkpoint format is little-endian"
#endif

namespace {

constexpr char kMagic[8] = {'Z', 'S', 'C', 'K', 'P', 'T', '0', '1'};
constexpr uint32_t kVersion = 1;
constexpr int32_t kArrays = 3;
constexpr int64_t kBlock = 1 << 20;        // bytes per checksummed block (written)
constexpr int64_t kUnit = 64 << 20;        // bytes staged per pipeline item
constexpr int64_t kPiece = 4 << 20;        // bytes per read-and-check task of a load
constexpr int64_t kPage = 4096;
constexpr int kSlots = 3;                  // staging buffers in flight
constexpr uint32_t kMetaId = 0x10, kHeaderId = 0x11;  // array ids of the small hashes
const char* const kArrayName[kArrays] = {"master", "exp_avg", "exp_avg_sq"};

struct Header {
  char magic[8];
  uint32_t version;
  int32_t layout;
  int32_t world, rank, n_params, n_arrays;
  int64_t P, P_pad, S, align, step;
  int64_t block_bytes, data_offset, array_stride, table_offset, file_bytes;
  uint64_t meta_hash;
  uint64_t header_hash;  // of the bytes before this field
};
static_assert(sizeof(Header) == 128, "checkpoint header is 128 bytes");

int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }
int64_t n_blocks(int64_t bytes, int64_t B) { return (bytes + B - 1) / B; }

// The block checksum of block_hash.h, on the host.
uint64_t host_hash(const unsigned char* p, int64_t len, int64_t block, int64_t B, uint32_t id) {
  const uint64_t base = zs::hash_base(id, block, B);
  uint64_t acc = zs::hash_seed(len, id);
  int64_t w = 0;
  for (; w + 8 <= len; w += 8) {
    uint64_t word;
    std::memcpy(&word, p + w, 8);
    acc += zs::hash_word(word, base + (uint64_t)(w / 8) + 1);
  }
  if (w < len) {
    uint64_t word = 0;
    for (int k = 0; w + k < len; ++k) word |= (uint64_t)p[w + k] << (8 * k);
    acc += zs::hash_word(word, base + (uint64_t)(w / 8) + 1);
  }
  return acc;
}

uint64_t header_hash_of(const Header& h) {
  return host_hash(reinterpret_cast<const unsigned char*>(&h), offsetof(Header, header_hash), 0,
                   kBlock, kHeaderId);
}

// A fixed set of worker threads for one call; run(n, f) runs f(0..n-1) on the
// workers and the caller and returns when all are done.
class Pool {
 public:
  explicit Pool(int n) {
    for (int i = 0; i + 1 < n; ++i) threads_.emplace_back([this] { loop(); });
  }
  ~Pool() {
    {
      std::lock_guard<std::mutex> l(mu_);
      stop_ = true;
    }
    cv_.notify_all();
    for (auto& t : threads_) t.join();
  }
  void run(int64_t n, const std::function<void(int64_t)>& f) {
    if (n <= 0) return;
    if (threads_.empty() || n == 1) {
      for (int64_t i = 0; i < n; ++i) f(i);
      return;
    }
    {
      std::lock_guard<std::mutex> l(mu_);
      job_ = &f;
      n_ = n;
      next_.store(0);
      busy_ = threads_.size();
      ++gen_;
    }
    cv_.notify_all();
    work();
    std::unique_lock<std::mutex> l(mu_);
    done_.wait(l, [this] { return busy_ == 0; });
    job_ = nullptr;
  }

 private:
  void work() {
    for (;;) {
      const int64_t i = next_.fetch_add(1);
      if (i >= n_) return;
      (*job_)(i);
    }
  }
  void loop() {
    uint64_t seen = 0;
    for (;;) {
      {
        std::unique_lock<std::mutex> l(mu_);
        cv_.wait(l, [&] { return stop_ || gen_ != seen; });
        if (stop_) return;
        seen = gen_;
      }
      work();
      std::lock_guard<std::mutex> l(mu_);
      if (--busy_ == 0) done_.notify_one();
    }
  }
  std::vector<std::thread> threads_;
  std::mutex mu_;
  std::condition_variable cv_, done_;
  const std::function<void(int64_t)>* job_ = nullptr;
  int64_t n_ = 0;
  std::atomic<int64_t> next_{0};
  size_t busy_ = 0;
  uint64_t gen_ = 0;
  bool stop_ = false;
};

int pool_threads() {
  const unsigned hw = std::thread::hardware_concurrency();
  return hw == 0 ? 4 : (int)std::min<unsigned>(hw, 16);
}

bool pread_full(int fd, void* buf, int64_t bytes, int64_t off) {
  unsigned char* p = static_cast<unsigned char*>(buf);
  while (bytes > 0) {
    const ssize_t r = pread(fd, p, (size_t)std::min<int64_t>(bytes, 1 << 30), (off_t)off);
    if (r < 0 && errno == EINTR) continue;
    if (r <= 0) return false;
    p += r;
    off += r;
    bytes -= r;
  }
  return true;
}

bool pwrite_full(int fd, const void* buf, int64_t bytes, int64_t off) {
  const unsigned char* p = static_cast<const unsigned char*>(buf);
  while (bytes > 0) {
    const ssize_t r = pwrite(fd, p, (size_t)std::min<int64_t>(bytes, 1 << 30), (off_t)off);
    if (r < 0 && errno == EINTR) continue;
    if (r <= 0) return false;
    p += r;
    off += r;
    bytes -= r;
  }
  return true;
}

// Buffered writes to one file: ext4 serialises writers of a file on its
// inode lock, and on the hosts measured one writer issuing 64 MiB pwrites into
// a preallocated file was the fastest (9 GB/s into the page cache, against
// about 7 GB/s for 2 to 16 writers), so a save has one writer thread.
bool write_pieces(int fd, const unsigned char* buf, int64_t bytes, int64_t off) {
  for (int64_t b0 = 0; b0 < bytes; b0 += kUnit)
    if (!pwrite_full(fd, buf + b0, std::min(kUnit, bytes - b0), off + b0)) return false;
  return true;
}

struct Fd {
  int fd = -1;
  Fd() = default;
  Fd(const Fd&) = delete;
  Fd& operator=(const Fd&) = delete;
  ~Fd() {
    if (fd >= 0) close(fd);
  }
};

// Where the elements of each parameter live in one layout.
struct Layout {
  int32_t kind = 0, world = 1;
  int64_t S = 0, P = 0;
  std::vector<int64_t> numels, offsets, rows, row_elems;
  std::vector<int32_t> owner;
  int32_t n() const { return (int32_t)numels.size(); }
  // Elements of a rows-layout parameter on each rank but the last.
  int64_t span(int32_t i) const { return rows[i] * row_elems[i]; }
};

Layout layout_of(const zs_plan* p) {
  Layout L;
  L.kind = p->layout;
  L.world = p->world;
  L.S = p->S;
  L.P = p->P;
  L.numels = p->numels;
  L.offsets = p->offsets;
  L.owner = p->owner;
  if (p->layout == zs::kLayoutRows) {
    L.rows = p->rows_per_rank;
    L.row_elems = p->row_elems;
  } else {
    L.rows.assign(p->n_params, 0);
    L.row_elems.assign(p->n_params, 0);
  }
  return L;
}

int64_t meta_bytes(int32_t n) { return (int64_t)n * 32 + round_up((int64_t)n * 4, 8); }

std::vector<unsigned char> encode_meta(const Layout& L) {
  const size_t n = (size_t)L.n();
  std::vector<unsigned char> out((size_t)meta_bytes(L.n()), 0);
  unsigned char* q = out.data();
  for (const std::vector<int64_t>* v : {&L.numels, &L.offsets, &L.rows, &L.row_elems}) {
    if (n) std::memcpy(q, v->data(), n * 8);
    q += n * 8;
  }
  for (size_t i = 0; i < n; ++i) {
    const int32_t tie = L.owner[i] == (int32_t)i ? -1 : L.owner[i];
    std::memcpy(q + 4 * i, &tie, 4);
  }
  return out;
}

void decode_meta(const unsigned char* q, int32_t n, Layout* L) {
  for (std::vector<int64_t>* v : {&L->numels, &L->offsets, &L->rows, &L->row_elems}) {
    v->resize(n);
    if (n) std::memcpy(v->data(), q, (size_t)n * 8);
    q += (size_t)n * 8;
  }
  L->owner.resize(n);
  for (int32_t i = 0; i < n; ++i) {
    int32_t tie;
    std::memcpy(&tie, q + 4 * (size_t)i, 4);
    L->owner[i] = tie < 0 ? i : tie;
  }
}

// A layout read from a file must place every element inside its ranks'
// arrays: then no index computed from it leaves a shard.
bool layout_sane(const Layout& L) {
  if (L.world < 1 || L.world > ZS_MAX_WORLD || L.S < 0) return false;
  if (L.S > INT64_MAX / 4 / L.world) return false;
  for (int32_t i = 0; i < L.n(); ++i) {
    const int64_t n = L.numels[i], off = L.offsets[i];
    if (n < 0 || off < 0 || L.owner[i] < 0 || L.owner[i] > i) return false;
    if (L.owner[i] != i) {
      if (L.owner[L.owner[i]] != L.owner[i] || L.numels[L.owner[i]] != n) return false;
      continue;
    }
    if (L.kind == zs::kLayoutFlat) {
      if (n > 0 && L.S == 0) return false;
      if (off > (int64_t)L.world * L.S - n) return false;
    } else {
      const int64_t r = L.rows[i], re = L.row_elems[i];
      if (r < 0 || re < 0) return false;
      if (n == 0) continue;
      if (re == 0 || r == 0 || r > L.S / re || r * re > L.S - off) return false;
      if ((n + r * re - 1) / (r * re) > L.world) return false;
    }
  }
  return true;
}

// The part of parameter i on rank r: elements [*e0, *e1) at local index *at.
void piece_of(const Layout& L, int32_t r, int32_t i, int64_t* e0, int64_t* e1, int64_t* at) {
  const int64_t n = L.numels[i];
  if (L.kind == zs::kLayoutFlat) {
    const int64_t off = L.offsets[i], lo = (int64_t)r * L.S;
    const int64_t a = std::max(off, lo), b = std::min(off + n, lo + L.S);
    *e0 = a - off;
    *e1 = std::max(a, b) - off;
    *at = a - lo;
  } else {
    const int64_t sp = L.span(i);
    *e0 = std::min((int64_t)r * sp, n);
    *e1 = std::min((int64_t)(r + 1) * sp, n);
    *at = L.offsets[i];
  }
}

// The rank holding element e of parameter i, its local index there, and the
// end of the run of elements from e that stay on that rank.
void locate(const Layout& L, int32_t i, int64_t e, int64_t* k, int64_t* at, int64_t* end) {
  const int64_t n = L.numels[i];
  if (L.kind == zs::kLayoutFlat) {
    const int64_t g = L.offsets[i] + e;
    *k = g / L.S;
    *at = g - *k * L.S;
    *end = std::min(n, (*k + 1) * L.S - L.offsets[i]);
  } else {
    const int64_t sp = L.span(i);
    *k = e / sp;
    *at = L.offsets[i] + e - *k * sp;
    *end = std::min(n, (*k + 1) * sp);
  }
}

struct Run {
  int64_t k, src, dst, len;  // old rank, old local index, new local index, elements
};

// Element runs of new rank r's shard and where each comes from.
std::vector<Run> build_runs(const Layout& nw, int32_t r, const Layout& old) {
  std::vector<Run> runs;
  for (int32_t i = 0; i < nw.n(); ++i) {
    if (nw.owner[i] != i) continue;
    int64_t e0, e1, at;
    piece_of(nw, r, i, &e0, &e1, &at);
    for (int64_t e = e0; e < e1;) {
      int64_t k, src, end;
      locate(old, i, e, &k, &src, &end);
      const int64_t take = std::min(e1, end) - e;
      const int64_t dst = at + (e - e0);
      if (!runs.empty() && runs.back().k == k && runs.back().src + runs.back().len == src &&
          runs.back().dst + runs.back().len == dst) {
        runs.back().len += take;
      } else {
        runs.push_back({k, src, dst, take});
      }
      e += take;
    }
  }
  return runs;
}

struct Copy {
  int64_t stage, dst, bytes;  // byte offsets: in the staged unit, in the new array
};
struct Unit {
  int64_t k, blk_lo, blk_hi;
  std::vector<Copy> copies;
};

// Staged reads: whole blocks of one old file, at most unit_blocks at a time,
// each listing the byte copies into the new shard that it feeds.
std::vector<Unit> make_units(std::vector<Run> runs, int64_t B, int64_t unit_blocks) {
  std::sort(runs.begin(), runs.end(), [](const Run& a, const Run& b) {
    return a.k != b.k ? a.k < b.k : a.src < b.src;
  });
  std::vector<Unit> units;
  for (const Run& r : runs) {
    int64_t s0 = r.src * 4, d = r.dst * 4;
    const int64_t s1 = (r.src + r.len) * 4;
    while (s0 < s1) {
      const int64_t blk = s0 / B;
      if (units.empty() || units.back().k != r.k || blk > units.back().blk_hi ||
          blk >= units.back().blk_lo + unit_blocks)
        units.push_back({r.k, blk, blk, {}});
      Unit& u = units.back();
      const int64_t e = std::min(s1, (u.blk_lo + unit_blocks) * B);
      u.copies.push_back({s0 - u.blk_lo * B, d, e - s0});
      u.blk_hi = std::max(u.blk_hi, n_blocks(e, B));
      d += e - s0;
      s0 = e;
    }
  }
  return units;
}

// Host or device memory, as the state arrays are. With no CUDA device, host.
enum class Mem { kHost, kDevice, kMixed };

Mem memory_of(void* const* ptrs, int n) {
  int kinds = 0;
  for (int i = 0; i < n; ++i) {
    if (!ptrs[i]) continue;
    cudaPointerAttributes attr;
    bool dev = false;
    if (cudaPointerGetAttributes(&attr, ptrs[i]) == cudaSuccess)
      dev = attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged;
    else
      cudaGetLastError();
    kinds |= dev ? 2 : 1;
  }
  return kinds == 3 ? Mem::kMixed : kinds == 2 ? Mem::kDevice : Mem::kHost;
}

zs_status check_state(const char* fn, int64_t S, void* const* arrays, bool output, Mem* mem) {
  const int64_t bytes = S * 4;
  for (int a = 0; a < kArrays; ++a)
    if (S > 0 && !arrays[a]) return zs::fail(ZS_ERR_INVAL, "%s: %s is NULL", fn, kArrayName[a]);
  *mem = memory_of(arrays, kArrays);
  if (*mem == Mem::kMixed)
    return zs::fail(ZS_ERR_INVAL, "%s: master, exp_avg and exp_avg_sq must all be host or all be "
                    "device memory", fn);
  if (S == 0) return ZS_OK;
  for (int a = 0; a < kArrays; ++a) {
    if (*mem == Mem::kDevice) {
      if (((uintptr_t)arrays[a] & 15u) != 0)
        return zs::fail(ZS_ERR_ALIGN, "%s: %s is not 16-byte aligned", fn, kArrayName[a]);
      if (zs_status st = zs::check_device_array(arrays[a], bytes, fn, kArrayName[a])) return st;
    }
    if (!output) continue;
    for (int b = 0; b < kArrays; ++b) {
      const uintptr_t x = (uintptr_t)arrays[a], y = (uintptr_t)arrays[b];
      if (a != b && x < y + (uint64_t)bytes && y < x + (uint64_t)bytes)
        return zs::fail(ZS_ERR_INVAL, "%s: %s overlaps %s", fn, kArrayName[a], kArrayName[b]);
    }
  }
  return ZS_OK;
}

// Pinned staging kept from one checkpoint call to the next: allocating and
// pinning kSlots x 64 MiB costs about 8 ms on a Grace host (measured), close
// to a tenth of a restore from the page cache. One set is kept (the last one
// returned, for one device and size); zs_checkpoint_release_staging frees it.
struct StagingCache {
  std::mutex mu;
  unsigned char* buf[kSlots] = {};  // guarded by mu; buf[0] == NULL: empty
  int64_t bytes = 0;
  int dev = -1;
};
StagingCache& staging_cache() {
  static StagingCache* c = new StagingCache;  // never destroyed: no CUDA calls at exit
  return *c;
}

// Staging buffers (pinned for device-resident state) and their events.
struct Staging {
  unsigned char* buf[kSlots] = {};
  cudaEvent_t ev[kSlots] = {};
  bool pinned = false;
  int64_t bytes = 0;
  int dev = -1;
  std::vector<unsigned char> host;
  Staging() = default;
  Staging(const Staging&) = delete;
  Staging& operator=(const Staging&) = delete;
  ~Staging() {
    for (int s = 0; s < kSlots; ++s)
      if (ev[s]) cudaEventDestroy(ev[s]);
    if (!pinned) return;
    bool all = true;
    for (int s = 0; s < kSlots; ++s) all = all && buf[s];
    if (all) {
      StagingCache& c = staging_cache();
      std::lock_guard<std::mutex> l(c.mu);
      if (!c.buf[0]) {  // keep this set for the next call
        for (int s = 0; s < kSlots; ++s) c.buf[s] = buf[s];
        c.bytes = bytes;
        c.dev = dev;
        return;
      }
    }
    for (int s = 0; s < kSlots; ++s)
      if (buf[s]) cudaFreeHost(buf[s]);
  }
  zs_status init(bool device, int64_t n, const char* fn) {
    if (!device) {
      try {
        host.resize((size_t)n * kSlots);
      } catch (...) {
        return zs::fail(ZS_ERR_NOMEM, "%s: no host memory for %lld bytes of staging", fn,
                        (long long)(n * kSlots));
      }
      for (int s = 0; s < kSlots; ++s) buf[s] = host.data() + (size_t)n * s;
      return ZS_OK;
    }
    pinned = true;
    bytes = n;
    if (cudaGetDevice(&dev) != cudaSuccess)
      return zs::fail(ZS_ERR_CUDA, "%s: staging: no current device", fn);
    {
      StagingCache& c = staging_cache();
      std::lock_guard<std::mutex> l(c.mu);
      if (c.buf[0] && c.bytes == n && c.dev == dev) {
        for (int s = 0; s < kSlots; ++s) {
          buf[s] = c.buf[s];
          c.buf[s] = nullptr;
        }
      }
    }
    for (int s = 0; s < kSlots; ++s) {
      cudaError_t e = cudaSuccess;
      if (!buf[s])
        e = cudaHostAlloc(reinterpret_cast<void**>(&buf[s]), (size_t)n, cudaHostAllocDefault);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev[s], cudaEventDisableTiming);
      if (e != cudaSuccess)
        return zs::fail(ZS_ERR_CUDA, "%s: staging: %s", fn, cudaGetErrorString(e));
    }
    return ZS_OK;
  }
};

zs_status cuda_fail(const char* fn, const char* what, cudaError_t e) {
  return zs::fail(ZS_ERR_CUDA, "%s: %s: %s", fn, what, cudaGetErrorString(e));
}

// Reads and checks the header of an open checkpoint file.
zs_status read_header(int fd, const char* path, Header* h, const char* fn) {
  struct stat st;
  if (fstat(fd, &st) != 0) return zs::fail(ZS_ERR_IO, "%s: cannot stat %s", fn, path);
  if (st.st_size < (off_t)sizeof(Header) || !pread_full(fd, h, sizeof *h, 0))
    return zs::fail(ZS_ERR_CORRUPT, "%s: %s is shorter than a checkpoint header", fn, path);
  if (std::memcmp(h->magic, kMagic, 8) != 0)
    return zs::fail(ZS_ERR_CORRUPT, "%s: %s is not a checkpoint shard", fn, path);
  if (h->version != kVersion)
    return zs::fail(ZS_ERR_CORRUPT, "%s: %s has format version %u, this library reads %u", fn,
                    path, h->version, kVersion);
  if (h->header_hash != header_hash_of(*h))
    return zs::fail(ZS_ERR_CORRUPT, "%s: %s: header checksum mismatch", fn, path);
  const int64_t B = h->block_bytes;
  const bool ok = (h->layout == zs::kLayoutFlat || h->layout == zs::kLayoutRows) &&
                  h->world >= 1 && h->world <= ZS_MAX_WORLD && h->rank >= 0 &&
                  h->rank < h->world && h->n_params >= 0 && h->n_arrays == kArrays &&
                  h->S >= 0 && h->S <= (INT64_MAX / 64) && h->step >= 0 && B >= 4096 &&
                  B <= (int64_t(1) << 30) && (B & (B - 1)) == 0 &&
                  h->data_offset >= (int64_t)sizeof(Header) + meta_bytes(h->n_params) &&
                  h->array_stride >= h->S * 4 &&
                  h->table_offset >= h->data_offset + kArrays * h->array_stride &&
                  h->file_bytes == h->table_offset + kArrays * n_blocks(h->S * 4, B) * 8;
  if (!ok) return zs::fail(ZS_ERR_CORRUPT, "%s: %s: inconsistent header fields", fn, path);
  if ((int64_t)st.st_size != h->file_bytes)
    return zs::fail(ZS_ERR_CORRUPT, "%s: %s has %lld bytes, its header says %lld (truncated?)", fn,
                    path, (long long)st.st_size, (long long)h->file_bytes);
  return ZS_OK;
}

}  // namespace

static zs_status zs_checkpoint_save_untraced(const zs_plan* plan, int32_t rank, const float* master,
                                        const float* exp_avg, const float* exp_avg_sq,
                                        int64_t step, const char* path, void* cuda_stream) {
  static const char* fn = "zs_checkpoint_save";
  zs::clear_error();
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "%s: not a live plan", fn);
  if (rank < 0 || rank >= plan->world)
    return zs::fail(ZS_ERR_RANGE, "%s: rank %d not in [0, %d)", fn, rank, plan->world);
  if (step < 0) return zs::fail(ZS_ERR_RANGE, "%s: step %lld < 0", fn, (long long)step);
  if (!path || !*path) return zs::fail(ZS_ERR_INVAL, "%s: path is NULL or empty", fn);
  void* arrays[kArrays] = {const_cast<float*>(master), const_cast<float*>(exp_avg),
                           const_cast<float*>(exp_avg_sq)};
  Mem mem;
  if (zs_status st = check_state(fn, plan->S, arrays, false, &mem)) return st;
  const bool device = mem == Mem::kDevice;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

  std::vector<unsigned char> meta;
  try {
    meta = encode_meta(layout_of(plan));
  } catch (...) {
    return zs::fail(ZS_ERR_NOMEM, "%s: out of host memory", fn);
  }
  const int64_t S = plan->S, bytes = S * 4, nb = n_blocks(bytes, kBlock);
  Header h;
  std::memset(&h, 0, sizeof h);
  std::memcpy(h.magic, kMagic, 8);
  h.version = kVersion;
  h.layout = plan->layout;
  h.world = plan->world;
  h.rank = rank;
  h.n_params = plan->n_params;
  h.n_arrays = kArrays;
  h.P = plan->P;
  h.P_pad = plan->P_pad;
  h.S = S;
  h.align = plan->align;
  h.step = step;
  h.block_bytes = kBlock;
  h.data_offset = round_up((int64_t)sizeof h + (int64_t)meta.size(), kPage);
  h.array_stride = round_up(bytes, kPage);
  h.table_offset = h.data_offset + kArrays * h.array_stride;
  h.file_bytes = h.table_offset + kArrays * nb * 8;
  h.meta_hash = host_hash(meta.data(), (int64_t)meta.size(), 0, kBlock, kMetaId);
  h.header_hash = header_hash_of(h);

  // Block checksums: on the device (per-block partial sums into mapped pinned
  // memory, added up once the stream is done), or on the host.
  std::vector<uint64_t> host_table;
  try {
    host_table.resize((size_t)(kArrays * nb));
  } catch (...) {
    return zs::fail(ZS_ERR_NOMEM, "%s: out of host memory", fn);
  }
  uint64_t* table = host_table.data();
  uint64_t* partials = nullptr;
  struct PinnedFree {
    void* p = nullptr;
    ~PinnedFree() {
      if (p) cudaFreeHost(p);
    }
  } partials_guard;
  const int parts = device && nb > 0 ? zs::block_hash_parts(nb, kBlock) : 1;
  if (device && nb > 0) {
    cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&partials),
                                  (size_t)(kArrays * nb * parts * 8), cudaHostAllocMapped);
    if (e != cudaSuccess) return cuda_fail(fn, "checksum table", e);
    partials_guard.p = partials;
    uint64_t* dpartials = nullptr;
    e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&dpartials), partials, 0);
    for (int a = 0; a < kArrays && e == cudaSuccess; ++a)
      e = zs::launch_block_hash(arrays[a], bytes, 0, kBlock, (uint32_t)a, parts,
                                dpartials + a * nb * parts, stream);
    if (e != cudaSuccess) {
      cudaStreamSynchronize(stream);
      return cuda_fail(fn, "checksum kernel", e);
    }
  } else if (nb > 0) {
    Pool pool(pool_threads());
    pool.run(kArrays * nb, [&](int64_t j) {
      const int64_t a = j / nb, b = j % nb, off = b * kBlock;
      table[j] = host_hash(static_cast<const unsigned char*>(arrays[a]) + off,
                           std::min(kBlock, bytes - off), b, kBlock, (uint32_t)a);
    });
  }

  // Written under a temporary name and renamed, so the final name never holds
  // a torn file.
  const std::string tmp = std::string(path) + ".part";
  Fd f;
  f.fd = open(tmp.c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
  if (f.fd < 0) {
    const int err = errno;
    if (device) cudaStreamSynchronize(stream);
    return zs::fail(ZS_ERR_IO, "%s: cannot create %s: %s", fn, tmp.c_str(), strerror(err));
  }
  // Ends a failed save: nothing left in flight, no partial file left behind.
  auto abandon = [&]() {
    if (device) cudaStreamSynchronize(stream);
    close(f.fd);
    f.fd = -1;
    std::remove(tmp.c_str());
  };
  auto io_fail = [&](const char* what) {
    abandon();
    return zs::fail(ZS_ERR_IO, "%s: %s %s failed", fn, what, tmp.c_str());
  };
  // Allocate the file's blocks up front (where the file system can): the
  // writes then fill allocated space instead of growing the file.
  const int fa = posix_fallocate(f.fd, 0, (off_t)h.file_bytes);
  if (fa != 0 && fa != EOPNOTSUPP && fa != EINVAL) return io_fail("allocating");
  std::vector<unsigned char> head(sizeof h + meta.size());
  std::memcpy(head.data(), &h, sizeof h);
  if (!meta.empty()) std::memcpy(head.data() + sizeof h, meta.data(), meta.size());
  if (!pwrite_full(f.fd, head.data(), (int64_t)head.size(), 0))
    return io_fail("writing the header of");

  if (!device) {
    for (int a = 0; a < kArrays; ++a)
      if (!write_pieces(f.fd, static_cast<const unsigned char*>(arrays[a]), bytes,
                        h.data_offset + a * h.array_stride))
        return io_fail("writing");
  } else if (bytes > 0) {
    // Items of kUnit bytes of one array; the device-to-host copies of the next
    // items run while one is written.
    Staging stg;
    if (zs_status st = stg.init(true, kUnit, fn)) {
      abandon();
      return st;
    }
    const int64_t per = n_blocks(bytes, kUnit), items = kArrays * per;
    auto enqueue = [&](int64_t i) {
      const int s = (int)(i % kSlots);
      const int64_t a = i / per, off = (i % per) * kUnit, len = std::min(kUnit, bytes - off);
      cudaError_t e = cudaMemcpyAsync(stg.buf[s], static_cast<unsigned char*>(arrays[a]) + off,
                                      (size_t)len, cudaMemcpyDeviceToHost, stream);
      if (e == cudaSuccess) e = cudaEventRecord(stg.ev[s], stream);
      return e;
    };
    cudaError_t e = cudaSuccess;
    for (int64_t i = 0; i < std::min<int64_t>(items, kSlots) && e == cudaSuccess; ++i)
      e = enqueue(i);
    for (int64_t i = 0; i < items && e == cudaSuccess; ++i) {
      const int s = (int)(i % kSlots);
      e = cudaEventSynchronize(stg.ev[s]);
      if (e != cudaSuccess) break;
      const int64_t a = i / per, off = (i % per) * kUnit, len = std::min(kUnit, bytes - off);
      if (!pwrite_full(f.fd, stg.buf[s], len, h.data_offset + a * h.array_stride + off))
        return io_fail("writing");
      if (i + kSlots < items) e = enqueue(i + kSlots);
    }
    if (e != cudaSuccess) {
      abandon();
      return cuda_fail(fn, "copy to host", e);
    }
  }
  if (device) {
    const cudaError_t e = cudaStreamSynchronize(stream);  // the partial sums are complete
    if (e != cudaSuccess) {
      abandon();
      return cuda_fail(fn, "stream", e);
    }
    for (int64_t j = 0; partials && j < kArrays * nb; ++j) {
      uint64_t sum = 0;
      for (int p = 0; p < parts; ++p) sum += partials[j * parts + p];
      table[j] = sum;
    }
  }
  if (nb > 0 && !pwrite_full(f.fd, table, kArrays * nb * 8, h.table_offset))
    return io_fail("writing the checksums of");
  if (ftruncate(f.fd, (off_t)h.file_bytes) != 0) return io_fail("sizing");
  const int rc = close(f.fd);
  f.fd = -1;
  if (rc != 0) {
    std::remove(tmp.c_str());
    return zs::fail(ZS_ERR_IO, "%s: closing %s failed", fn, tmp.c_str());
  }
  if (std::rename(tmp.c_str(), path) != 0) {
    const int err = errno;
    std::remove(tmp.c_str());
    return zs::fail(ZS_ERR_IO, "%s: cannot rename %s to %s: %s", fn, tmp.c_str(), path,
                    strerror(err));
  }
  return ZS_OK;
}

extern "C" zs_status zs_checkpoint_info(const char* path, int32_t* world, int32_t* rank,
                                        int32_t* layout, int32_t* n_params, int64_t* P,
                                        int64_t* S, int64_t* step) {
  static const char* fn = "zs_checkpoint_info";
  zs::clear_error();
  if (!path) return zs::fail(ZS_ERR_INVAL, "%s: path is NULL", fn);
  Fd f;
  f.fd = open(path, O_RDONLY);
  if (f.fd < 0) return zs::fail(ZS_ERR_IO, "%s: cannot open %s: %s", fn, path, strerror(errno));
  Header h;
  if (zs_status st = read_header(f.fd, path, &h, fn)) return st;
  if (world) *world = h.world;
  if (rank) *rank = h.rank;
  if (layout) *layout = h.layout;
  if (n_params) *n_params = h.n_params;
  if (P) *P = h.P;
  if (S) *S = h.S;
  if (step) *step = h.step;
  return ZS_OK;
}

static zs_status zs_checkpoint_load_untraced(const zs_plan* plan, int32_t rank,
                                        const char* const* paths, int32_t n_paths, float* master,
                                        float* exp_avg, float* exp_avg_sq, int64_t* step,
                                        void* cuda_stream) {
  static const char* fn = "zs_checkpoint_load";
  zs::clear_error();
  if (!zs::plan_is_live(plan)) return zs::fail(ZS_ERR_INVAL, "%s: not a live plan", fn);
  if (rank < 0 || rank >= plan->world)
    return zs::fail(ZS_ERR_RANGE, "%s: rank %d not in [0, %d)", fn, rank, plan->world);
  if (!paths || n_paths < 1 || n_paths > ZS_MAX_WORLD)
    return zs::fail(ZS_ERR_INVAL, "%s: need the old ranks' files (1..%d paths)", fn,
                    ZS_MAX_WORLD);
  if (!paths[0]) return zs::fail(ZS_ERR_INVAL, "%s: paths[0] (old rank 0) is NULL", fn);
  void* arrays[kArrays] = {master, exp_avg, exp_avg_sq};
  Mem mem;
  if (zs_status st = check_state(fn, plan->S, arrays, true, &mem)) return st;
  const bool device = mem == Mem::kDevice;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

  // Old rank 0's file fixes the old layout; it must hold this parameter list.
  std::vector<Fd> files(n_paths);
  Header h0;
  files[0].fd = open(paths[0], O_RDONLY);
  if (files[0].fd < 0)
    return zs::fail(ZS_ERR_IO, "%s: cannot open %s: %s", fn, paths[0], strerror(errno));
  if (zs_status st = read_header(files[0].fd, paths[0], &h0, fn)) return st;
  if (h0.rank != 0 || h0.world != n_paths)
    return zs::fail(ZS_ERR_CORRUPT, "%s: %s is rank %d of %d; expected rank 0 of %d", fn,
                    paths[0], h0.rank, h0.world, n_paths);
  if (h0.n_params != plan->n_params || h0.P != plan->P)
    return zs::fail(ZS_ERR_INVAL, "%s: %s holds %d parameters (%lld elements), the plan %d "
                    "(%lld)", fn, paths[0], h0.n_params, (long long)h0.P, plan->n_params,
                    (long long)plan->P);
  const int64_t mb = meta_bytes(h0.n_params);
  std::vector<unsigned char> meta0((size_t)mb);
  if (mb > 0 && !pread_full(files[0].fd, meta0.data(), mb, sizeof(Header)))
    return zs::fail(ZS_ERR_IO, "%s: reading %s failed", fn, paths[0]);
  if (host_hash(meta0.data(), mb, 0, kBlock, kMetaId) != h0.meta_hash)
    return zs::fail(ZS_ERR_CORRUPT, "%s: %s: metadata checksum mismatch", fn, paths[0]);
  Layout old;
  old.kind = h0.layout;
  old.world = h0.world;
  old.S = h0.S;
  old.P = h0.P;
  decode_meta(meta0.data(), h0.n_params, &old);
  for (int32_t i = 0; i < plan->n_params; ++i)
    if (old.numels[i] != plan->numels[i] || old.owner[i] != plan->owner[i])
      return zs::fail(ZS_ERR_INVAL, "%s: parameter %d of %s (%lld elements, stored with %d) "
                      "differs from the plan's (%lld, %d)", fn, i, paths[0],
                      (long long)old.numels[i], old.owner[i], (long long)plan->numels[i],
                      plan->owner[i]);
  if (!layout_sane(old))
    return zs::fail(ZS_ERR_CORRUPT, "%s: %s: its layout does not fit its shards", fn, paths[0]);

  std::vector<Run> runs;
  try {
    runs = build_runs(layout_of(plan), rank, old);
  } catch (...) {
    return zs::fail(ZS_ERR_NOMEM, "%s: out of host memory", fn);
  }
  const int64_t B = h0.block_bytes, ob = h0.S * 4, onb = n_blocks(ob, B);
  std::vector<std::vector<uint64_t>> tables(n_paths);
  std::vector<char> needed(n_paths, 0);
  for (const Run& r : runs) needed[r.k] = 1;
  for (int32_t k = 0; k < n_paths; ++k) {
    if (!needed[k]) continue;
    if (k > 0) {
      if (!paths[k])
        return zs::fail(ZS_ERR_INVAL, "%s: rank %d needs old rank %d's file; paths[%d] is NULL",
                        fn, rank, k, k);
      files[k].fd = open(paths[k], O_RDONLY);
      if (files[k].fd < 0)
        return zs::fail(ZS_ERR_IO, "%s: cannot open %s: %s", fn, paths[k], strerror(errno));
      Header h;
      if (zs_status st = read_header(files[k].fd, paths[k], &h, fn)) return st;
      if (h.rank != k || h.world != n_paths)
        return zs::fail(ZS_ERR_CORRUPT, "%s: %s is rank %d of %d; expected rank %d of %d", fn,
                        paths[k], h.rank, h.world, k, n_paths);
      if (h.layout != h0.layout || h.S != h0.S || h.P != h0.P || h.n_params != h0.n_params ||
          h.block_bytes != B || h.meta_hash != h0.meta_hash || h.data_offset != h0.data_offset ||
          h.array_stride != h0.array_stride || h.table_offset != h0.table_offset)
        return zs::fail(ZS_ERR_CORRUPT, "%s: %s and %s describe different layouts", fn,
                        paths[k], paths[0]);
      if (h.step != h0.step)
        return zs::fail(ZS_ERR_CORRUPT, "%s: %s is at step %lld, %s at step %lld", fn, paths[k],
                        (long long)h.step, paths[0], (long long)h0.step);
      std::vector<unsigned char> meta((size_t)mb);
      if (mb > 0 && (!pread_full(files[k].fd, meta.data(), mb, sizeof(Header)) || meta != meta0))
        return zs::fail(ZS_ERR_CORRUPT, "%s: %s: metadata differs from %s's", fn, paths[k],
                        paths[0]);
    }
    tables[k].resize((size_t)(kArrays * onb));
    if (onb > 0 &&
        !pread_full(files[k].fd, tables[k].data(), kArrays * onb * 8, h0.table_offset))
      return zs::fail(ZS_ERR_IO, "%s: reading the checksums of %s failed", fn, paths[k]);
  }

  // The new shard's padding (elements no run writes) becomes zero.
  std::vector<Run> by_dst = runs;
  std::sort(by_dst.begin(), by_dst.end(), [](const Run& a, const Run& b) { return a.dst < b.dst; });
  std::vector<std::pair<int64_t, int64_t>> gaps;  // [lo, hi) in elements
  int64_t at = 0;
  for (const Run& r : by_dst) {
    if (r.dst > at) gaps.push_back({at, r.dst});
    at = std::max(at, r.dst + r.len);
  }
  if (at < plan->S) gaps.push_back({at, plan->S});
  if (device) {
    std::vector<zs::RowSegment> segs;
    for (int a = 0; a < kArrays; ++a)
      for (const auto& g : gaps)
        segs.push_back({nullptr, static_cast<unsigned char*>(arrays[a]) + g.first * 4, 0,
                        (g.second - g.first) * 4});
    if (!segs.empty()) {
      const cudaError_t e = zs::launch_segment_copy(segs.data(), (int)segs.size(), stream);
      if (e != cudaSuccess) {
        cudaStreamSynchronize(stream);
        return cuda_fail(fn, "zero fill", e);
      }
    }
  } else {
    for (int a = 0; a < kArrays; ++a)
      for (const auto& g : gaps)
        std::memset(static_cast<unsigned char*>(arrays[a]) + g.first * 4, 0,
                    (size_t)(g.second - g.first) * 4);
  }

  const int64_t unit_blocks = std::max<int64_t>(1, kUnit / B);
  std::vector<Unit> units;
  try {
    units = make_units(runs, B, unit_blocks);
  } catch (...) {
    if (device) cudaStreamSynchronize(stream);
    return zs::fail(ZS_ERR_NOMEM, "%s: out of host memory", fn);
  }
  // Which blocks the device checks: those lying whole inside one copy whose
  // destination is 16-byte aligned (all of a same-layout restore but a ragged
  // last one; all but the edge blocks of each run of a resharding one). The
  // hash kernel reads them where they landed in HBM, so for them the host
  // only reads the file; every other block read is hashed on the host.
  struct Span {
    int64_t dst, fb0, fb1;  // destination byte of block fb0; blocks [fb0, fb1)
    int64_t slot;           // first of its (fb1 - fb0) * parts partial sums
    int parts;
  };
  std::vector<std::vector<Span>> spans(units.size());
  std::vector<std::vector<char>> host_check(units.size());
  int64_t n_dev = 0;  // partial sums of the device-checked blocks, per array
  try {
    for (size_t ui = 0; ui < units.size(); ++ui) {
      const Unit& u = units[ui];
      host_check[ui].assign((size_t)(u.blk_hi - u.blk_lo), 1);
      if (!device) continue;
      for (const Copy& c : u.copies) {
        const int64_t src0 = u.blk_lo * B + c.stage, src1 = src0 + c.bytes;
        const int64_t fb0 = n_blocks(src0, B);
        const int64_t fb1 = src1 == ob ? n_blocks(ob, B) : src1 / B;
        if (fb1 <= fb0) continue;
        const int64_t dst = c.dst + (fb0 * B - src0);
        if (dst % 16 != 0) continue;
        const int parts = zs::block_hash_parts(fb1 - fb0, B);
        spans[ui].push_back({dst, fb0, fb1, n_dev, parts});
        n_dev += (fb1 - fb0) * parts;
        for (int64_t b = fb0; b < fb1; ++b) host_check[ui][(size_t)(b - u.blk_lo)] = 0;
      }
    }
  } catch (...) {
    if (device) cudaStreamSynchronize(stream);
    return zs::fail(ZS_ERR_NOMEM, "%s: out of host memory", fn);
  }
  uint64_t* dev_sums = nullptr;  // mapped pinned: [kArrays][n_dev]
  uint64_t* dev_sums_d = nullptr;
  struct PinnedFree {
    void* p = nullptr;
    ~PinnedFree() {
      if (p) cudaFreeHost(p);
    }
  } sums_guard;
  if (n_dev > 0) {
    cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&dev_sums),
                                  (size_t)(kArrays * n_dev * 8), cudaHostAllocMapped);
    if (e == cudaSuccess) {
      sums_guard.p = dev_sums;
      e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&dev_sums_d), dev_sums, 0);
    }
    if (e != cudaSuccess) {
      cudaStreamSynchronize(stream);
      return cuda_fail(fn, "checksum table", e);
    }
  }
  Staging stg;
  if (zs_status st = stg.init(device, unit_blocks * B, fn)) {
    if (device) cudaStreamSynchronize(stream);
    return st;
  }
  Pool pool(pool_threads());
  const int64_t items = (int64_t)units.size() * kArrays;
  const int64_t piece_blocks = std::max<int64_t>(1, kPiece / B);
  // Every (item, piece) is one task of one pool run, items in order (item i =
  // array i % 3 of unit i / 3), so the next items' reads go on while an
  // item's last pieces finish: no barrier per item. Item i stages in slot
  // i % kSlots once item i - kSlots has left it (issued, and on the device
  // its copies done); the task that reads an item's last piece issues, in
  // item order, the copies of every item that is then complete.
  std::vector<int64_t> first((size_t)items + 1, 0);
  for (int64_t i = 0; i < items; ++i) {
    const Unit& u = units[(size_t)(i / kArrays)];
    first[(size_t)i + 1] = first[(size_t)i] + n_blocks(u.blk_hi - u.blk_lo, piece_blocks);
  }
  std::mutex mu;
  std::condition_variable cv;
  std::vector<int64_t> left((size_t)items);  // guarded by mu: pieces not yet read
  for (int64_t i = 0; i < items; ++i)
    left[(size_t)i] = first[(size_t)i + 1] - first[(size_t)i];
  std::vector<char> issued((size_t)items, 0);  // guarded by mu
  int64_t next_issue = 0;                      // guarded by mu
  bool stop = false;                           // guarded by mu: a failure; tasks return
  bool io_bad = false;
  int64_t bad_block = -1;
  int bad_k = 0, bad_a = 0;
  cudaError_t cuda_bad = cudaSuccess;
  int dev = 0;
  if (device && cudaGetDevice(&dev) != cudaSuccess) {
    cudaStreamSynchronize(stream);
    return zs::fail(ZS_ERR_CUDA, "%s: no current device", fn);
  }
  // Copies item i out of its slot (device: enqueued, with the checksums of
  // the blocks the device checks and the slot's event). Called with mu held.
  auto issue = [&](int64_t i) -> cudaError_t {
    const size_t ui = (size_t)(i / kArrays);
    const Unit& u = units[ui];
    const int a = (int)(i % kArrays);
    const int s = (int)(i % kSlots);
    unsigned char* out = static_cast<unsigned char*>(arrays[a]);
    if (!device) {
      for (const Copy& c : u.copies)
        std::memcpy(out + c.dst, stg.buf[s] + c.stage, (size_t)c.bytes);
      return cudaSuccess;
    }
    cudaError_t e = cudaSuccess;
    for (const Copy& c : u.copies) {
      e = cudaMemcpyAsync(out + c.dst, stg.buf[s] + c.stage, (size_t)c.bytes,
                          cudaMemcpyHostToDevice, stream);
      if (e != cudaSuccess) return e;
    }
    for (const Span& sp : spans[ui]) {
      e = zs::launch_block_hash(out + sp.dst, std::min(sp.fb1 * B, ob) - sp.fb0 * B, sp.fb0, B,
                                (uint32_t)a, sp.parts, dev_sums_d + a * n_dev + sp.slot,
                                stream);
      if (e != cudaSuccess) return e;
    }
    return cudaEventRecord(stg.ev[s], stream);
  };
  pool.run(first[(size_t)items], [&](int64_t p) {
    const int64_t i =
        (int64_t)(std::upper_bound(first.begin(), first.end(), p) - first.begin()) - 1;
    const size_t ui = (size_t)(i / kArrays);
    const Unit& u = units[ui];
    const int a = (int)(i % kArrays);
    const int s = (int)(i % kSlots);
    if (device) cudaSetDevice(dev);  // worker threads: the caller's device
    if (i >= kSlots) {
      std::unique_lock<std::mutex> l(mu);
      cv.wait(l, [&] { return stop || issued[(size_t)(i - kSlots)]; });
      if (stop) return;
    } else {
      std::lock_guard<std::mutex> l(mu);
      if (stop) return;
    }
    if (device && i >= kSlots) {
      // The slot's last user's copies (its event is not recorded again before
      // this item's pieces are all read).
      const cudaError_t e = cudaEventSynchronize(stg.ev[s]);
      if (e != cudaSuccess) {
        std::lock_guard<std::mutex> l(mu);
        stop = true;
        cuda_bad = e;
        cv.notify_all();
        return;
      }
    }
    // Read this piece's blocks and check the ones the host checks.
    const int64_t base = h0.data_offset + a * h0.array_stride;
    const int64_t b0 = u.blk_lo + (p - first[(size_t)i]) * piece_blocks;
    const int64_t b1 = std::min(u.blk_hi, b0 + piece_blocks);
    const int64_t off = b0 * B, len = std::min(b1 * B, ob) - off;
    unsigned char* dst = stg.buf[s] + (off - u.blk_lo * B);
    bool read_ok = pread_full(files[(size_t)u.k].fd, dst, len, base + off);
    int64_t bad = -1;
    for (int64_t b = b0; read_ok && b < b1 && bad < 0; ++b) {
      if (!host_check[ui][(size_t)(b - u.blk_lo)]) continue;
      const int64_t l = std::min(B, ob - b * B);
      if (host_hash(dst + (b - b0) * B, l, b, B, (uint32_t)a) !=
          tables[(size_t)u.k][(size_t)(a * onb + b)])
        bad = b;
    }
    std::lock_guard<std::mutex> l(mu);
    if (!read_ok || bad >= 0) {
      if (!stop) {
        io_bad = !read_ok;
        bad_block = bad;
        bad_k = u.k;
        bad_a = a;
      }
      stop = true;
      cv.notify_all();
      return;
    }
    if (--left[(size_t)i] > 0 || stop) return;
    while (next_issue < items && left[(size_t)next_issue] == 0) {
      const cudaError_t e = issue(next_issue);
      if (e != cudaSuccess) {
        stop = true;
        cuda_bad = e;
        break;
      }
      issued[(size_t)next_issue] = 1;
      ++next_issue;
    }
    cv.notify_all();
  });
  // Items without pieces (none in practice) are issued here.
  while (!stop && next_issue < items) {
    const cudaError_t e = issue(next_issue++);
    if (e != cudaSuccess) {
      stop = true;
      cuda_bad = e;
    }
  }
  if (stop) {
    if (device) cudaStreamSynchronize(stream);
    if (io_bad) return zs::fail(ZS_ERR_IO, "%s: reading %s failed", fn, paths[bad_k]);
    if (bad_block >= 0)
      return zs::fail(ZS_ERR_CORRUPT, "%s: %s: %s block %lld checksum mismatch (the state "
                      "arrays now hold partial data)", fn, paths[bad_k], kArrayName[bad_a],
                      (long long)bad_block);
    return cuda_fail(fn, "copy to device", cuda_bad);
  }
  if (device) {
    const cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(fn, "stream", e);
    for (size_t ui = 0; ui < units.size(); ++ui)
      for (const Span& sp : spans[ui])
        for (int a = 0; a < kArrays; ++a)
          for (int64_t b = sp.fb0; b < sp.fb1; ++b) {
            uint64_t sum = 0;
            const uint64_t* part = dev_sums + a * n_dev + sp.slot + (b - sp.fb0) * sp.parts;
            for (int p = 0; p < sp.parts; ++p) sum += part[p];
            if (sum != tables[(size_t)units[ui].k][(size_t)(a * onb + b)])
              return zs::fail(ZS_ERR_CORRUPT, "%s: %s: %s block %lld checksum mismatch (the "
                              "state arrays now hold partial data)", fn, paths[units[ui].k],
                              kArrayName[a], (long long)b);
          }
  }
  if (step) *step = h0.step;
  return ZS_OK;
}

// ---- traced entry points ----------------------------------------------------------
extern "C" zs_status zs_checkpoint_save(const zs_plan* plan, int32_t rank, const float* master,
                                        const float* exp_avg, const float* exp_avg_sq,
                                        int64_t step, const char* path, void* cuda_stream) {
  const zs::CallRange range("zs_checkpoint_save");
  return zs::traced(zs_checkpoint_save_untraced(plan, rank, master, exp_avg, exp_avg_sq, step,
                                                path, cuda_stream),
                    "zs_checkpoint_save", plan, rank, 0, 0, -1, -1, step);
}

extern "C" zs_status zs_checkpoint_load(const zs_plan* plan, int32_t rank,
                                        const char* const* paths, int32_t n_paths, float* master,
                                        float* exp_avg, float* exp_avg_sq, int64_t* step,
                                        void* cuda_stream) {
  const zs::CallRange range("zs_checkpoint_load");
  int64_t saved = -1;
  const zs_status st = zs_checkpoint_load_untraced(plan, rank, paths, n_paths, master, exp_avg,
                                                   exp_avg_sq, &saved, cuda_stream);
  if (st == ZS_OK && step) *step = saved;
  return zs::traced(st, "zs_checkpoint_load", plan, rank, 0, 0, -1, -1, saved);
}

extern "C" zs_status zs_checkpoint_release_staging(void) {
  zs::clear_error();
  StagingCache& c = staging_cache();
  std::lock_guard<std::mutex> l(c.mu);
  cudaError_t first = cudaSuccess;
  for (int s = 0; s < kSlots; ++s) {
    if (!c.buf[s]) continue;
    const cudaError_t e = cudaFreeHost(c.buf[s]);
    if (first == cudaSuccess) first = e;
    c.buf[s] = nullptr;
  }
  c.bytes = 0;
  c.dev = -1;
  if (first != cudaSuccess)
    return zs::fail(ZS_ERR_CUDA, "zs_checkpoint_release_staging: %s", cudaGetErrorString(first));
  return ZS_OK;
}
