// The C ABI (include/nspack.h): host-side checks, table allocation through
// the caller's allocator, and the order of kernel launches that builds a
// context and assembles updates.  No packing arithmetic runs on the host: the
// host only validates arguments, sizes tables, reads back the few scalars it
// needs to size the next ones, and estimates from the weights where the held-
// out hash's first round may stop before the quotas are known (a scheduling
// hint that no result depends on).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <utility>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "nspack.h"

struct ns_pack_ctx {
  // recipe
  uint32_t T = 0, B = 0, K = 0, flags = 0, S = 0, J = 0, n_docs = 0, G = 0, len_bucket = 0;
  int32_t pad_id = 0;
  uint64_t seed = 0, hash_key = 0, n_tokens = 0;
  const int32_t *tokens = nullptr;
  int32_t *tokens_rw = nullptr;  // the context's own copy of a host-resident corpus
  const int64_t *offs = nullptr;
  const int32_t *loss_start = nullptr;
  cudaStream_t stream = nullptr;
  ns_alloc_fn alloc = nullptr;
  ns_free_fn free_fn = nullptr;
  void *user = nullptr;
  int n_sms = 0;
  // host summary
  std::vector<uint32_t> piece_begin, piece_B;  // the schedule (one piece without one)
  std::vector<uint64_t> windows;
  std::vector<uint8_t> complete;
  uint32_t valid_steps = 0, levels = 0, init_launches = 0;
  uint64_t digest = 0, n_pieces = 0, table_bytes = 0;
  uint64_t host_bytes = 0;  // bytes of a host-resident corpus read at init
  uint64_t hashed_tokens = 0, hashed_docs = 0;  // what the held-out hash read at init
  uint64_t hash_ns = 0;                          // its device time
  bool speculate = true;    // hash to a bound speculated from the measured fill
  uint32_t init_passes = 1;
  // device tables kept for the per-update calls
  int32_t *rb = nullptr, *cum = nullptr, *quota = nullptr;
  uint32_t *W = nullptr;
  int64_t *wbase = nullptr;
  int4 *row_win = nullptr;
  int64_t *node_S = nullptr, *node_src = nullptr;
  int32_t *node_doc = nullptr, *node_mthr = nullptr;
  int *err = nullptr;
  uint64_t *fp_out = nullptr;
  uint64_t *pad_tail = nullptr;
  std::vector<void *> kept;
  int device = 0;                  // the device the tables live on
  std::atomic<bool> foreign{false};  // a step ran on a stream other than `stream`
};

namespace {

void dev_free(ns_pack_ctx *c, void *p) {
  if (!p) return;
  if (c->free_fn)
    c->free_fn(p, c->user);
  else
    cudaFree(p);
}

// Page-locked host memory for the small copies of an init (the grid layouts
// and estimates it uploads, its two readbacks): a copy from pageable memory
// goes through a driver buffer and may wait for the stream; one from
// page-locked memory is a plain DMA.  One buffer per host thread, grown at
// the start of an init when it is too small -- no copy of an earlier init is
// in flight then, as every init synchronises its streams before it returns
// -- and handed out front to back during the init.  Ordinary memory stands
// in if page-locked memory cannot be had.
struct HostStage {
  char *pinned = nullptr;
  std::vector<char> heap;
  size_t cap = 0, used = 0;
  void reset(size_t need) {
    used = 0;
    if (need <= cap) return;
    if (pinned) cudaFreeHost(pinned);
    pinned = nullptr;
    const size_t c = std::max<size_t>(need, (size_t)1 << 20);
    void *p = nullptr;
    if (cudaHostAlloc(&p, c, cudaHostAllocPortable) == cudaSuccess) {
      pinned = static_cast<char *>(p);
      std::vector<char>().swap(heap);
    } else {
      cudaGetLastError();
      heap.resize(c);
    }
    cap = c;
  }
  void *take(size_t bytes) {  // NULL past what the init reserved
    const size_t off = (used + 255) / 256 * 256;
    if (off + bytes > cap) return nullptr;
    used = off + bytes;
    return (pinned ? pinned : heap.data()) + off;
  }
  ~HostStage() {
    if (pinned) cudaFreeHost(pinned);
  }
};
thread_local HostStage tl_stage;

// Device memory of one init.  Small requests are carved out of slabs that
// grow geometrically (1 MiB, 2 MiB, ... up to 64 MiB), large ones get their
// own allocation, so an init makes a handful of allocator calls instead of
// one per table.  Tables the context keeps and temporaries of the init come
// from separate slabs; the temporaries go back when the init ends.
struct Arena {
  struct Slab {
    char *base = nullptr;
    size_t size = 0, used = 0, next = 1u << 20;
  };
  static constexpr size_t kMaxSlab = 64u << 20;
  ns_pack_ctx *c;
  std::vector<void *> temps;
  Slab keep_slab, temp_slab;
  explicit Arena(ns_pack_ctx *ctx) : c(ctx) {}
  void *raw(size_t bytes, bool keep) {
    void *p = nullptr;
    if (c->alloc) {
      p = c->alloc(bytes, c->user);
    } else if (cudaMalloc(&p, bytes) != cudaSuccess) {
      cudaGetLastError();
      p = nullptr;
    }
    if (!p) return nullptr;
    if (keep) {
      c->kept.push_back(p);
      c->table_bytes += bytes;
    } else {
      temps.push_back(p);
    }
    return p;
  }
  void *get(size_t bytes, bool keep) {
    bytes = ((bytes + 255) / 256) * 256;
    if (bytes == 0) bytes = 256;
    Slab &s = keep ? keep_slab : temp_slab;
    if (s.base && s.used + bytes <= s.size) {
      void *p = s.base + s.used;
      s.used += bytes;
      return p;
    }
    if (bytes * 2 > s.next) return raw(bytes, keep);  // large: its own allocation
    char *b = static_cast<char *>(raw(s.next, keep));
    if (!b) return nullptr;
    s.base = b;
    s.size = s.next;
    s.used = bytes;
    s.next = std::min(s.next * 2, kMaxSlab);
    return b;
  }
  // Room for `bytes` more (the sum of the coming arrays, each rounded up to
  // 256) in one allocation: a phase of the init makes one call of the
  // allocation callback instead of one per large array.  What does not fit
  // after all is allocated as before.
  bool reserve(size_t bytes, bool keep) {
    Slab &s = keep ? keep_slab : temp_slab;
    if (bytes == 0 || (s.base && s.size - s.used >= bytes)) return true;
    char *b = static_cast<char *>(raw(bytes, keep));
    if (!b) return false;
    s.base = b;
    s.size = bytes;
    s.used = 0;
    return true;
  }
  static size_t rounded(size_t bytes) { return bytes ? (bytes + 255) / 256 * 256 : 256; }
  template <class T>
  T *keep(size_t n) {
    return static_cast<T *>(get(n * sizeof(T), true));
  }
  template <class T>
  T *temp(size_t n) {
    return static_cast<T *>(get(n * sizeof(T), false));
  }
  // Host memory for a copy of this init: the thread's page-locked stage, or,
  // past what the init reserved of it, ordinary memory kept until the init
  // ends.
  std::vector<std::vector<char>> host_extra;
  void *host(size_t bytes) {
    void *p = tl_stage.take(bytes);
    if (p) return p;
    host_extra.emplace_back(std::max<size_t>(bytes, 1));
    return host_extra.back().data();
  }
  void release() {
    for (void *p : temps) dev_free(c, p);
    temps.clear();
    temp_slab = Slab();
  }
};

void release_ctx(ns_pack_ctx *c) {
  if (!c) return;
  for (void *p : c->kept) dev_free(c, p);
  c->kept.clear();
  delete c;
}

// A device pointer aligned for its element type: the kernels' loads and
// stores of that type would fault on a misaligned one.
template <class T>
bool aligned_for(const T *p) {
  return reinterpret_cast<uintptr_t>(p) % alignof(T) == 0;
}

int check_config(const ns_pack_config *cfg) {
  if (!cfg || !cfg->tokens || !cfg->doc_offsets) return NS_ERR_INVALID_ARG;
  if (!cfg->stream_doc_begin || !cfg->stream_source || !cfg->source_weight ||
      !cfg->stream_weight || !cfg->source_heldout_bp)
    return NS_ERR_INVALID_ARG;
  if (!(cfg->flags & NS_PACK_HOST_CORPUS) &&
      (reinterpret_cast<uintptr_t>(cfg->tokens) % 16 != 0 || !aligned_for(cfg->doc_offsets) ||
       !aligned_for(cfg->loss_start)))
    return NS_ERR_INVALID_ARG;
  if (cfg->T < 16 || cfg->T % 16 != 0 || cfg->T > NS_MAX_T) return NS_ERR_INVALID_ARG;
  if (cfg->B == 0 || cfg->max_steps == 0) return NS_ERR_INVALID_ARG;
  if ((uint64_t)cfg->max_steps * cfg->B >= (1ull << 31)) return NS_ERR_INVALID_ARG;
  if (cfg->n_docs >= (1u << 31)) return NS_ERR_INVALID_ARG;
  if (cfg->n_tokens >= NS_MAX_TOKENS) return NS_ERR_INVALID_ARG;
  if (cfg->n_sources == 0 || cfg->n_sources > NS_MAX_SOURCES) return NS_ERR_INVALID_ARG;
  if (cfg->n_streams == 0 || cfg->n_streams > NS_MAX_STREAMS) return NS_ERR_INVALID_ARG;
  if (cfg->flags & ~(NS_PACK_DRAIN | NS_PACK_HELDOUT | NS_PACK_SHUFFLE_ROWS | NS_PACK_WRAP |
                     NS_PACK_HOST_CORPUS | NS_PACK_ORDERED_FREE))
    return NS_ERR_INVALID_ARG;
  if (cfg->window_segment > NS_MAX_WINDOW_SEGMENT) return NS_ERR_INVALID_ARG;
  if ((cfg->alloc == nullptr) != (cfg->free == nullptr)) return NS_ERR_INVALID_ARG;
  if ((cfg->flags & NS_PACK_ORDERED_FREE) && !cfg->free) return NS_ERR_INVALID_ARG;
  for (uint32_t s = 0; s < cfg->n_sources; s++)
    if (cfg->source_weight[s] == 0 || cfg->source_heldout_bp[s] > 10000) return NS_ERR_INVALID_ARG;
  std::vector<uint32_t> per_source(cfg->n_sources, 0);
  for (uint32_t j = 0; j < cfg->n_streams; j++) {
    if (cfg->stream_weight[j] == 0 || cfg->stream_source[j] >= cfg->n_sources)
      return NS_ERR_INVALID_ARG;
    if (j > 0 && cfg->stream_source[j] < cfg->stream_source[j - 1]) return NS_ERR_INVALID_ARG;
    if (cfg->stream_doc_begin[j + 1] < cfg->stream_doc_begin[j]) return NS_ERR_INVALID_ARG;
    per_source[cfg->stream_source[j]]++;
  }
  if (cfg->stream_doc_begin[cfg->n_streams] > cfg->n_docs) return NS_ERR_INVALID_ARG;
  for (uint32_t s = 0; s < cfg->n_sources; s++)
    if (per_source[s] == 0 || per_source[s] > NS_MAX_STRATA_PER_SOURCE) return NS_ERR_INVALID_ARG;
  if (cfg->n_pieces) {
    if (!cfg->piece_begin || !cfg->piece_B || !cfg->piece_source_weight ||
        !cfg->piece_stream_weight)
      return NS_ERR_INVALID_ARG;
    if (cfg->n_pieces > cfg->max_steps || cfg->piece_begin[0] != 0) return NS_ERR_INVALID_ARG;
    for (uint32_t p = 0; p < cfg->n_pieces; p++) {
      if (p > 0 && cfg->piece_begin[p] <= cfg->piece_begin[p - 1]) return NS_ERR_INVALID_ARG;
      if (cfg->piece_begin[p] >= cfg->max_steps) return NS_ERR_INVALID_ARG;
      if (cfg->piece_B[p] == 0 || cfg->piece_B[p] > cfg->B) return NS_ERR_INVALID_ARG;
      for (uint32_t s = 0; s < cfg->n_sources; s++)
        if (cfg->piece_source_weight[(size_t)p * cfg->n_sources + s] == 0)
          return NS_ERR_INVALID_ARG;
      for (uint32_t j = 0; j < cfg->n_streams; j++)
        if (cfg->piece_stream_weight[(size_t)p * cfg->n_streams + j] == 0)
          return NS_ERR_INVALID_ARG;
    }
  }
  return NS_OK;
}

// Rows of update k (the schedule's piece's, or B).
uint32_t rows_of_step(const ns_pack_ctx *c, uint32_t k) {
  size_t p = 0;
  for (size_t q = 0; q < c->piece_begin.size(); q++)
    if (c->piece_begin[q] <= k) p = q;
  return c->piece_B[p];
}

// Block layout of a segmented launch: count[j] items per stream, `per`
// items per block.
std::vector<uint32_t> seg_layout(const std::vector<uint64_t> &count, uint32_t per) {
  std::vector<uint32_t> base(count.size() + 1, 0);
  uint64_t acc = 0;
  for (size_t j = 0; j < count.size(); j++) {
    base[j] = (uint32_t)acc;
    acc += (count[j] + per - 1) / per;
  }
  base[count.size()] = (uint32_t)acc;
  return base;
}

#define NS_CK(x)                                 \
  do {                                           \
    if ((x) != cudaSuccess) {                    \
      cudaGetLastError();                        \
      return NS_ERR_CUDA;                        \
    }                                            \
  } while (0)
#define NS_ALLOC(p)               \
  do {                            \
    if (!(p)) return NS_ERR_OOM;  \
  } while (0)

// A second stream for work that does not depend on the corpus, with its fork
// and join events; synchronised on every exit path.  Created once per host
// thread and device and kept for the next init (creating a stream and its
// events costs more than a small init's kernels).
struct SideHandles {
  cudaStream_t s = nullptr, s2 = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, join2 = nullptr;
  cudaEvent_t t0 = nullptr, t1 = nullptr;  // timing: the held-out hash's phase
};
constexpr int kMaxSideDevices = 64;
// The handles of one host thread, released when the thread ends (errors
// ignored: at process exit the runtime may already be gone).
struct SidePool {
  SideHandles h[kMaxSideDevices];
  ~SidePool() {
    for (SideHandles &x : h) {
      for (cudaEvent_t e : {x.fork, x.join, x.join2, x.t0, x.t1})
        if (e) cudaEventDestroy(e);
      if (x.s) cudaStreamDestroy(x.s);
      if (x.s2) cudaStreamDestroy(x.s2);
    }
    cudaGetLastError();
  }
};
thread_local SidePool tl_side;

struct SideStream {
  cudaStream_t s = nullptr, s2 = nullptr;  // two: the quotas, the offsets check
  cudaEvent_t fork = nullptr, join = nullptr, join2 = nullptr, t0 = nullptr, t1 = nullptr;
  cudaError_t create() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    SideHandles local, *h = (dev >= 0 && dev < kMaxSideDevices) ? &tl_side.h[dev] : &local;
    if (!h->s) {
      e = cudaStreamCreateWithFlags(&h->s, cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->fork, cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->join, cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->s2, cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->join2, cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreate(&h->t0);
      if (e == cudaSuccess) e = cudaEventCreate(&h->t1);
      if (e != cudaSuccess) {
        // release a partial set, so that the next init creates a whole one
        for (cudaEvent_t *ev : {&h->fork, &h->join, &h->join2, &h->t0, &h->t1})
          if (*ev) cudaEventDestroy(*ev), *ev = nullptr;
        for (cudaStream_t *q : {&h->s, &h->s2})
          if (*q) cudaStreamDestroy(*q), *q = nullptr;
        return e;
      }
    }
    s = h->s;
    s2 = h->s2;
    fork = h->fork;
    join = h->join;
    join2 = h->join2;
    t0 = h->t0;
    t1 = h->t1;
    owned = (h == &local);
    return cudaSuccess;
  }
  bool owned = false;  // a device beyond the table: destroyed with this object
  ~SideStream() {
    if (s) cudaStreamSynchronize(s);
    if (s2) cudaStreamSynchronize(s2);
    if (owned) {
      if (fork) cudaEventDestroy(fork);
      if (join) cudaEventDestroy(join);
      if (join2) cudaEventDestroy(join2);
      if (s2) cudaStreamDestroy(s2);
      if (t0) cudaEventDestroy(t0);
      if (t1) cudaEventDestroy(t1);
      if (s) cudaStreamDestroy(s);
    }
  }
};

// A corpus given in host memory: the context's own device copy, filled by a
// second stream in groups of whole streams so that the hash of one group runs
// while the next group is copied.
struct CorpusCopy {
  cudaStream_t s = nullptr;
  std::vector<cudaEvent_t> done;          // one per group, on s
  std::vector<uint32_t> j_first;          // group g holds streams [j_first[g], j_first[g+1])
  cudaError_t create() { return cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking); }
  cudaError_t add_group(const int32_t *host, int32_t *dev, uint64_t begin, uint64_t end) {
    cudaEvent_t e;
    cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (r != cudaSuccess) return r;
    done.push_back(e);
    if (end > begin)
      r = cudaMemcpyAsync(dev + begin, host + begin, (end - begin) * sizeof(int32_t),
                          cudaMemcpyHostToDevice, s);
    if (r == cudaSuccess) r = cudaEventRecord(e, s);
    return r;
  }
  ~CorpusCopy() {
    if (s) cudaStreamSynchronize(s);
    for (cudaEvent_t e : done) cudaEventDestroy(e);
    if (s) cudaStreamDestroy(s);
  }
};

// Host arrays gathered into one buffer and copied to the device in one call.
struct Staging {
  std::vector<unsigned char> host;
  std::vector<std::pair<size_t, void **>> slots;
  void add(const void *p, size_t bytes, void **dev) {
    const size_t off = (host.size() + 255) / 256 * 256;
    host.resize(off + std::max<size_t>(bytes, 1));
    if (bytes) std::memcpy(host.data() + off, p, bytes);
    slots.emplace_back(off, dev);
  }
  // One copy of everything added, into temporary memory of the init or, with
  // `keep`, into memory the context keeps.
  int commit(Arena &a, cudaStream_t st, bool keep = false) {
    unsigned char *d = static_cast<unsigned char *>(a.get(host.size(), keep));
    if (!d) return NS_ERR_OOM;
    void *h = a.host(host.size());
    std::memcpy(h, host.data(), host.size());
    if (cudaMemcpyAsync(d, h, host.size(), cudaMemcpyHostToDevice, st) != cudaSuccess) {
      cudaGetLastError();
      return NS_ERR_CUDA;
    }
    for (auto &s : slots) *s.second = d + s.first;
    return NS_OK;
  }
};

// Token bounds of every stream, ob[j] = doc_offsets[stream_doc_begin[j]],
// from the host offsets; false if they are not nondecreasing inside [0,
// n_tokens] (the device check then reports the partition).
bool stream_token_bounds(const ns_pack_config *cfg, uint32_t J, uint64_t nt,
                         std::vector<uint64_t> &ob) {
  ob.assign(J + 1, 0);
  for (uint32_t j = 0; j <= J; j++) {
    const int64_t v = cfg->doc_offsets[cfg->stream_doc_begin[j]];
    if (v < 0 || (uint64_t)v > nt || (j > 0 && (uint64_t)v < ob[j - 1])) return false;
    ob[j] = (uint64_t)v;
  }
  return true;
}

// The device address of n tokens in host memory when both ends of the range
// are page-locked memory the device can address (cudaHostAlloc, or
// registered with cudaHostRegister) and it starts on a 16-byte boundary;
// NULL otherwise (the corpus is then copied whole).
const int32_t *device_view(const int32_t *host, uint64_t n) {
  if (!host || n == 0) return nullptr;
  cudaPointerAttributes a0{}, a1{};
  if (cudaPointerGetAttributes(&a0, host) != cudaSuccess ||
      cudaPointerGetAttributes(&a1, host + (n - 1)) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a0.type != cudaMemoryTypeHost || a1.type != cudaMemoryTypeHost || !a0.devicePointer ||
      !a1.devicePointer)
    return nullptr;
  const char *d0 = static_cast<const char *>(a0.devicePointer);
  const char *d1 = static_cast<const char *>(a1.devicePointer);
  if (d1 - d0 != (ptrdiff_t)((n - 1) * sizeof(int32_t))) return nullptr;
  if (reinterpret_cast<uintptr_t>(d0) & 15) return nullptr;
  return reinterpret_cast<const int32_t *>(d0);
}

int upload(Arena &a, const void *host, size_t bytes, void **dev, cudaStream_t st) {
  *dev = a.get(bytes, false);
  NS_ALLOC(*dev);
  if (bytes) {
    void *h = a.host(bytes);
    std::memcpy(h, host, bytes);
    NS_CK(cudaMemcpyAsync(*dev, h, bytes, cudaMemcpyHostToDevice, st));
  }
  return NS_OK;
}

// build() asks to be run again with the full hash bound (internal, > 0).
constexpr int kRetryFullBound = 1;

// Builds every table of a context on cfg->cuda_stream, in this order:
//   host work and one upload: the recipe, the block layouts and estimates
//     the host knows, the reservation of this phase's arrays;
//   1./side streams: the quota tables (beside everything up to the cutoff),
//     the offsets check and the padding terms;
//   2. round keys and the shuffle of every stream (or of the estimated
//      prefix of a stream without a held-out rate);
//   3. the held-out hash of the prefix each stream's horizon reaches (two
//      rounds when the bound is speculated);
//   4. the scans of kept lengths and pieces, the cutoff, and the first
//      readback (its sizes decide what follows);
//   5. (host corpus) the tokens of the prefixes the hash did not read;
//   6. host work and the second upload; pieces, next-window search and
//      pointer jumping;
//   7. window counts and starts, the row table and the valid horizon;
//   8.-9. the order digest and the summary readback.
// Returns kRetryFullBound when a speculated bound left a stream short (the
// caller builds again with the full bound).
int build(ns_pack_ctx *c, const ns_pack_config *cfg, Arena &a) {
  const uint32_t J = c->J, S = c->S, K = c->K, T = c->T;
  cudaStream_t st = c->stream;
  {
    // this init's page-locked host memory: the recipe (a schedule's weights
    // up to 32 MiB; beyond, ordinary memory), the grid layouts and the two
    // readbacks, all proportional to the streams
    const size_t P = cfg->n_pieces ? cfg->n_pieces : 1;
    const size_t recipe = std::min<size_t>(P * ((size_t)S + J) * 12, (size_t)32 << 20);
    tl_stage.reset(recipe + 192 * ((size_t)J + 1) + 16 * ((size_t)S + 1) + ((size_t)256 << 10));
  }
  int dev = 0;
  NS_CK(cudaGetDevice(&dev));
  c->device = dev;
  NS_CK(cudaDeviceGetAttribute(&c->n_sms, cudaDevAttrMultiProcessorCount, dev));
  int rc;

  // ---- a corpus in host memory: the context's device copy ----------------
  // Offsets and loss starts first (the shuffle needs them).  Tokens in
  // page-locked memory the device can address are read where they lie: the
  // hash writes every document it reads into the copy and a copy kernel
  // brings over the reachable prefix of the streams it does not read, so
  // only the documents the horizon reaches cross the host link.  Other host
  // memory is copied whole, in groups of whole streams on a second stream,
  // the hash of each group waiting only for its own copy.
  const bool host_corpus = (c->flags & NS_PACK_HOST_CORPUS) != 0;
  const int32_t *htok = nullptr;  // device address of host tokens read in place
  CorpusCopy copy;
  if (host_corpus) {
    htok = device_view(cfg->tokens, c->n_tokens);
    int32_t *tok = a.keep<int32_t>(c->n_tokens + 4);
    int64_t *offs = a.keep<int64_t>((size_t)c->n_docs + 1);
    int32_t *ls = cfg->loss_start ? a.keep<int32_t>(std::max<uint32_t>(c->n_docs, 1)) : nullptr;
    NS_ALLOC(tok);
    NS_ALLOC(offs);
    if (cfg->loss_start) NS_ALLOC(ls);
    NS_CK(cudaMemcpyAsync(offs, cfg->doc_offsets, ((size_t)c->n_docs + 1) * 8,
                          cudaMemcpyHostToDevice, st));
    if (ls)
      NS_CK(cudaMemcpyAsync(ls, cfg->loss_start, (size_t)c->n_docs * 4, cudaMemcpyHostToDevice,
                            st));
    c->host_bytes = ((uint64_t)c->n_docs + 1) * 8 + (ls ? (uint64_t)c->n_docs * 4 : 0);
    if (!htok) {
      NS_CK(copy.create());
      // group boundaries where whole streams end, about an eighth of the
      // tokens each; offsets that are not nondecreasing inside [0, n_tokens]
      // at the streams' bounds make one group (the device check then reports
      // them)
      const uint64_t nt = c->n_tokens;
      std::vector<uint64_t> ob;
      const bool ok = stream_token_bounds(cfg, J, nt, ob);
      uint64_t begin = 0;
      copy.j_first.push_back(0);
      if (ok) {
        const uint64_t target = std::max<uint64_t>(nt / 8, 1);
        for (uint32_t j = 1; j < J; j++)
          if (ob[j] - begin >= target) {
            NS_CK(copy.add_group(cfg->tokens, tok, begin, ob[j]));
            copy.j_first.push_back(j);
            begin = ob[j];
          }
      }
      NS_CK(copy.add_group(cfg->tokens, tok, begin, nt));
      copy.j_first.push_back(J);
      c->host_bytes += nt * 4;
    }
    c->tokens = tok;
    c->tokens_rw = tok;
    c->offs = offs;
    c->loss_start = ls;
  }

  // ---- recipe tables on the device (temporaries) --------------------------
  std::vector<uint32_t> sdb(cfg->stream_doc_begin, cfg->stream_doc_begin + J + 1);
  std::vector<uint32_t> ssrc(cfg->stream_source, cfg->stream_source + J);
  std::vector<uint32_t> sw(cfg->source_weight, cfg->source_weight + S);
  std::vector<uint32_t> tw(cfg->stream_weight, cfg->stream_weight + J);
  std::vector<uint16_t> sbp(cfg->source_heldout_bp, cfg->source_heldout_bp + S);
  std::vector<uint16_t> stream_bp(J);
  std::vector<uint32_t> src_first(S + 1, 0);
  uint32_t max_strata = 0;
  bool any_heldout = false;
  for (uint32_t j = 0; j < J; j++) {
    stream_bp[j] = sbp[ssrc[j]];
    any_heldout |= stream_bp[j] > 0 && sdb[j + 1] > sdb[j];
  }
  for (uint32_t s = 0, j = 0; s < S; s++) {
    src_first[s] = j;
    while (j < J && ssrc[j] == s) j++;
    src_first[s + 1] = j;
    max_strata = std::max(max_strata, src_first[s + 1] - src_first[s]);
  }
  void *d_sdb, *d_ssrc, *d_sw, *d_tw, *d_sbp, *d_stream_bp, *d_src_first;
  Staging up;
  up.add(sdb.data(), sdb.size() * 4, &d_sdb);
  up.add(ssrc.data(), ssrc.size() * 4, &d_ssrc);
  up.add(sw.data(), sw.size() * 4, &d_sw);
  up.add(tw.data(), tw.size() * 4, &d_tw);
  up.add(sbp.data(), sbp.size() * 2, &d_sbp);
  up.add(stream_bp.data(), stream_bp.size() * 2, &d_stream_bp);
  up.add(src_first.data(), src_first.size() * 4, &d_src_first);
  // the schedule: one piece (B, the weights) without one
  const uint32_t P = cfg->n_pieces ? cfg->n_pieces : 1;
  std::vector<uint32_t> psw((size_t)P * S), ptw((size_t)P * J);
  if (cfg->n_pieces) {
    c->piece_begin.assign(cfg->piece_begin, cfg->piece_begin + P);
    c->piece_B.assign(cfg->piece_B, cfg->piece_B + P);
    psw.assign(cfg->piece_source_weight, cfg->piece_source_weight + (size_t)P * S);
    ptw.assign(cfg->piece_stream_weight, cfg->piece_stream_weight + (size_t)P * J);
  } else {
    c->piece_begin.assign(1, 0);
    c->piece_B.assign(1, c->B);
    psw = sw;
    ptw = tw;
  }
  void *d_pbegin, *d_pB, *d_psw, *d_ptw;
  up.add(c->piece_begin.data(), (size_t)P * 4, &d_pbegin);
  up.add(c->piece_B.data(), (size_t)P * 4, &d_pB);
  up.add(psw.data(), psw.size() * 4, &d_psw);
  up.add(ptw.data(), ptw.size() * 4, &d_ptw);
  // the schedule's digest items: count, then per piece begin, B, weights
  std::vector<uint64_t> piece_items;
  if (cfg->n_pieces) {
    piece_items.push_back(P);
    for (uint32_t p = 0; p < P; p++) {
      piece_items.push_back(c->piece_begin[p]);
      piece_items.push_back(c->piece_B[p]);
      for (uint32_t s2 = 0; s2 < S; s2++) piece_items.push_back(psw[(size_t)p * S + s2]);
      for (uint32_t j = 0; j < J; j++) piece_items.push_back(ptw[(size_t)p * J + j]);
    }
  }
  void *d_piece_items = nullptr;
  if (!piece_items.empty()) up.add(piece_items.data(), piece_items.size() * 8, &d_piece_items);

  // Each stream's windows over the horizon estimated from the recipe (its
  // share of every piece's rows, a few windows over): the quota rule keeps
  // every cumulative count within one window of its share.  Only how much of
  // a stream is shuffled and hashed before its exact need is known depends
  // on it.
  std::vector<double> est_windows(J, 0.0);
  for (uint32_t p = 0; p < P; p++) {
    const uint32_t kb = c->piece_begin[p];
    const uint32_t ke = (p + 1 < P) ? c->piece_begin[p + 1] : K;
    double swsum = 0.0;
    for (uint32_t s2 = 0; s2 < S; s2++) swsum += psw[(size_t)p * S + s2];
    for (uint32_t s2 = 0; s2 < S; s2++) {
      double twsum = 0.0;
      for (uint32_t j = src_first[s2]; j < src_first[s2 + 1]; j++) twsum += ptw[(size_t)p * J + j];
      for (uint32_t j = src_first[s2]; j < src_first[s2 + 1]; j++)
        est_windows[j] += (double)(ke - kb) * c->piece_B[p] * (psw[(size_t)p * S + s2] / swsum) *
                          (ptw[(size_t)p * J + j] / twsum);
    }
  }
  for (uint32_t j = 0; j < J; j++)
    est_windows[j] = std::ceil(est_windows[j]) + 2.0 + (c->G ? (double)c->G : 0.0);

  const uint32_t D0 = sdb[0];
  const uint64_t n_pos = (uint64_t)sdb[J] - D0;
  const bool heldout_mode = (c->flags & NS_PACK_HELDOUT) != 0;
  const bool wrap = (c->flags & NS_PACK_WRAP) != 0;
  std::vector<uint64_t> N(J);
  for (uint32_t j = 0; j < J; j++) N[j] = (uint64_t)sdb[j + 1] - sdb[j];
  // A stream without a held-out rate is shuffled, on the first pass, only
  // over about the positions its horizon needs (est_tok: the recipe's
  // estimate of its windows times T; see the shuffle below)
  bool any_unhashed = false;
  for (uint32_t j = 0; j < J; j++) any_unhashed |= stream_bp[j] == 0 && N[j] > 0;
  const bool shuffle_prefix = c->speculate && !heldout_mode && any_unhashed;
  std::vector<unsigned long long> est_tok;
  void *d_est = nullptr;
  if (shuffle_prefix) {
    est_tok.resize(J);
    for (uint32_t j = 0; j < J; j++) est_tok[j] = (unsigned long long)(est_windows[j] * T);
    up.add(est_tok.data(), J * sizeof(unsigned long long), &d_est);
  }
  // Two rounds of the hash only if some hashed stream may need enough
  // windows to be speculated at all (the recipe's estimate, which is within a
  // few windows of the quota table's; a stream below the threshold keeps the
  // full bound either way): else one round to the full bound, without the
  // fill kernel
  bool some_speculated = false;
  for (uint32_t j = 0; j < J; j++)
    some_speculated |= stream_bp[j] != 0 && est_windows[j] >= (double)nsk::kSpeculateMinWindows;
  const bool speculate = c->speculate && any_heldout && !wrap && some_speculated;
  // Until the quota kernel publishes each stream's need, the first round
  // stops a stream at half its recipe estimate (est_windows), not at no
  // bound at all: a small stream is then not hashed far past its need while
  // the quotas run.  A heuristic only: the second round hashes every stream
  // to its exact bound whatever the first one did.
  std::vector<unsigned long long> cap;
  void *d_cap = nullptr;
  if (speculate) {
    cap.resize(J);
    for (uint32_t j = 0; j < J; j++)
      cap[j] = (unsigned long long)(0.5 * est_windows[j] * (double)T);
    up.add(cap.data(), J * sizeof(unsigned long long), &d_cap);
  }
  // the shuffle's block layout
  const std::vector<uint32_t> order_bb = seg_layout(N, 256 * nsk::order_positions_per_thread());
  void *d_order_bb;
  up.add(order_bb.data(), order_bb.size() * 4, &d_order_bb);

  // What the host reads back after the prefix cutoff, in one block (one
  // copy): cutoff u32[J] | npieces i64[J] | node_base i64[J + 1] | ptokens
  // i64[J] | rmax i32[J] | need_num u16[J] | pos_lim u32[J] | error word
  auto al8 = [](size_t b) { return (b + 7) / 8 * 8; };
  const size_t r1_np = al8((size_t)J * 4), r1_nb = r1_np + (size_t)J * 8;
  const size_t r1_pt = r1_nb + ((size_t)J + 1) * 8, r1_rmax = r1_pt + (size_t)J * 8;
  const size_t r1_num = al8(r1_rmax + (size_t)J * 4), r1_lim = al8(r1_num + (size_t)J * 2);
  const size_t r1_err = r1_lim + (size_t)J * 4, r1_bytes = r1_err + 8;
  // The summary the host reads back at the end, in one block (one copy):
  // tokens read from host memory u64 | tokens and documents hashed u64[2] |
  // the digest's accumulator u64[2] | the first bad update (K - k) u32 |
  // order digest u64 | valid updates u32 | error word | windows u32[J]; its
  // first 48 bytes (counters and accumulators) start at zero
  constexpr size_t r2_read = 0, r2_hashed = 8, r2_dacc = 24, r2_bad = 40, r2_digest = 48;
  constexpr size_t r2_valid = 56, r2_err = 60, r2_W = 64;
  const size_t r2_bytes = r2_W + (size_t)J * 4;
  // One block of words that start at zero, cleared by one memset: the
  // quota kernel's ready count and the done counts of the kernels whose last
  // block finishes a step (the cutoff, the row table, the digest, the scans'
  // tile sums), then the
  // summary read back at the end (its counters and accumulators), then the
  // hash's per-stream frontier and progress words.
  constexpr size_t kCtlBytes = 256;
  const size_t zb_rb2 = kCtlBytes, zb_front = zb_rb2 + Arena::rounded(r2_bytes);
  const size_t zb_prog = zb_front + (any_heldout ? (size_t)J * 8 : 0);
  const size_t zb_bytes = zb_prog + (any_heldout ? (size_t)J * 8 : 0);
  const uint32_t n_tiles = (T + 127) / 128;
  const bool quota_warp = S <= 32 && max_strata <= 32;
  const size_t scan_bytes = nsk::scan_scratch_bytes(n_pos);
  {
    // the arrays of the phase up to the first readback, in one allocation
    // of each kind
    const auto R = Arena::rounded;
    const size_t n1 = std::max<uint64_t>(n_pos, 1);
    const size_t keep = R(sizeof(int)) + R(8) + R(((size_t)n_tiles + 1) * 8) +
                        R((size_t)K * J * 4) + R(((size_t)K + 1) * J * 4) +
                        R((size_t)K * (J + 1) * 4);
    const size_t temp = R(up.host.size()) + R((size_t)n_tiles * 8) + R(zb_bytes) +
                        (quota_warp ? 0 : R((size_t)K * S * 4)) + R((size_t)J * 32) +
                        2 * R(n1 * 4) + 2 * R((n_pos + 1) * 8) + R(scan_bytes) + R(r1_bytes);
    if (!a.reserve(keep, true) || !a.reserve(temp, false)) return NS_ERR_OOM;
  }
  if ((rc = up.commit(a, st))) return rc;
  if (piece_items.empty()) d_piece_items = nullptr;
  const nsk::QuotaPieces qp{static_cast<uint32_t *>(d_pbegin), static_cast<uint32_t *>(d_pB),
                            static_cast<uint32_t *>(d_psw), static_cast<uint32_t *>(d_ptw), P};

  c->err = a.keep<int>(1);
  NS_ALLOC(c->err);
  c->fp_out = a.keep<uint64_t>(1);
  NS_ALLOC(c->fp_out);
  // fingerprint terms of padding, per tile of a row, for the gather
  // (computed on the second side stream below)
  c->pad_tail = a.keep<uint64_t>(n_tiles + 1);
  uint64_t *pad_tiles = a.temp<uint64_t>(n_tiles);
  NS_ALLOC(c->pad_tail);
  NS_ALLOC(pad_tiles);
  NS_CK(cudaMemsetAsync(c->err, 0, sizeof(int), st));
  char *zb = a.temp<char>(zb_bytes);
  NS_ALLOC(zb);
  NS_CK(cudaMemsetAsync(zb, 0, zb_bytes, st));
  unsigned *ready = reinterpret_cast<unsigned *>(zb);
  unsigned *done_cutoff = ready + 1, *done_rows = ready + 2, *done_digest = ready + 3;
  unsigned *done_scan = ready + 4;
  char *rb2 = zb + zb_rb2;

  // ---- 1. quotas of every update, on a side stream ------------------------
  // They depend only on the weights, so they run while the corpus is hashed
  // and shuffled; the main stream joins them before the prefix cutoff.
  c->quota = a.keep<int32_t>((size_t)K * J);
  c->cum = a.keep<int32_t>((size_t)(K + 1) * J);
  c->rb = a.keep<int32_t>((size_t)K * (J + 1));
  NS_ALLOC(c->quota);
  NS_ALLOC(c->cum);
  NS_ALLOC(c->rb);
  SideStream side;
  NS_CK(side.create());
  // the side streams start from here (the recipe uploaded, the control block
  // zeroed); their launches are issued after the main stream's keys and
  // shuffle, which the host enqueues first
  NS_CK(cudaEventRecord(side.fork, st));

  // ---- 2. shuffled order and lengths of every position ----------------------
  uint64_t *keys = a.temp<uint64_t>((size_t)J * 4);
  uint32_t *order = a.temp<uint32_t>(std::max<uint64_t>(n_pos, 1));
  uint32_t *klen = a.temp<uint32_t>(std::max<uint64_t>(n_pos, 1));
  int64_t *kex = a.temp<int64_t>(n_pos + 1);
  int64_t *pex = a.temp<int64_t>(n_pos + 1);
  void *scan_scratch = a.get(scan_bytes, false);
  NS_ALLOC(keys);
  NS_ALLOC(order);
  NS_ALLOC(klen);
  NS_ALLOC(kex);
  NS_ALLOC(pex);
  NS_ALLOC(scan_scratch);
  // A stream without a held-out rate (nothing to hash) needs only the
  // shuffled positions whose documents hold its horizon's tokens: on the
  // first pass about that many are taken (a quarter over the recipe's
  // estimate); the others are not shuffled, and the shuffle gives length 0
  // to those the scans read.  A stream whose windows turn out to
  // need more is caught after the cutoff, and the context is built again
  // with every position.
  char *rb1 = a.temp<char>(r1_bytes);
  NS_ALLOC(rb1);
  uint32_t *pos_lim = nullptr;
  if (shuffle_prefix) pos_lim = reinterpret_cast<uint32_t *>(rb1 + r1_lim);
  NS_CK(nsk::launch_keys_bound(c->seed, J, keys, static_cast<uint32_t *>(d_sdb), c->offs,
                               static_cast<uint16_t *>(d_stream_bp),
                               static_cast<unsigned long long *>(d_est), pos_lim, st));
  {
    nsk::SegGrid g{static_cast<uint32_t *>(d_order_bb), J, order_bb[J]};
    NS_CK(nsk::launch_order(g, static_cast<uint32_t *>(d_sdb), keys, c->offs, c->n_tokens, D0,
                            heldout_mode ? static_cast<uint16_t *>(d_stream_bp) : nullptr,
                            pos_lim, order, klen, c->err, c->n_sms, st));
  }

  // ---- the side streams: quotas; the offsets check and padding terms ------
  NS_CK(cudaStreamWaitEvent(side.s, side.fork, 0));
  if (quota_warp) {
    NS_CK(nsk::launch_quota_warp(qp, S, static_cast<uint32_t *>(d_src_first), J, K, max_strata,
                                 c->quota, c->cum, ready, side.s));
  } else {
    int32_t *src_quota = a.temp<int32_t>((size_t)K * S);
    NS_ALLOC(src_quota);
    NS_CK(nsk::launch_quota_sources(qp, S, K, src_quota, side.s));
    NS_CK(nsk::launch_quota_strata(qp, src_quota, static_cast<uint32_t *>(d_src_first), S, J, K,
                                   max_strata, c->quota, c->cum, ready, side.s));
  }
  NS_CK(nsk::launch_row_base(c->quota, J, K, c->rb, side.s));
  NS_CK(cudaEventRecord(side.join, side.s));
  // The corpus partition, checked whole on a stream of its own beside the
  // quotas, the shuffle and the hash: every kernel that reads tokens also
  // checks the offsets it uses, so a malformed partition is reported
  // (BAD_INPUT) at the next readback, never read past.
  NS_CK(cudaStreamWaitEvent(side.s2, side.fork, 0));
  NS_CK(nsk::launch_validate_offsets(c->offs, c->n_docs, c->n_tokens, c->err, c->n_sms,
                                     side.s2));
  NS_CK(nsk::launch_pad_tail(c->pad_id, T, pad_tiles, c->pad_tail, side.s2));
  NS_CK(cudaEventRecord(side.join2, side.s2));

  // ---- 3. held-out flags of the prefix each stream's horizon reaches -------
  // Runs beside the quota kernels: it reads each stream's need from their
  // table once all S quota blocks have published it, and hashes on until then.
  // tokens read from host memory in place (hash and prefix copy)
  unsigned long long *tokens_read =
      htok ? reinterpret_cast<unsigned long long *>(rb2 + r2_read) : nullptr;
  const bool group_copy = host_corpus && !htok;
  // Greedy windows hold at most T tokens, so a prefix whose kept tokens
  // exceed (windows needed) * T holds them all, whatever the packing: the
  // full bound.  Greedy packing fills about four fifths of a window, so the
  // hash goes in two rounds instead: to half the bound, then -- once every
  // stream's fill has been measured on a sample of its decided documents --
  // to that fill plus a margin.  The packing then shows whether each prefix
  // holds the windows it must; if one does not, the context is built again
  // with the full bound.  Wrap packing fills every window: full bound.
  uint16_t *need_num = nullptr;  // per stream, of 1024 (NULL: the full bound)
  unsigned long long *pre_cap = nullptr;
  if (speculate) {
    need_num = reinterpret_cast<uint16_t *>(rb1 + r1_num);
    pre_cap = static_cast<unsigned long long *>(d_cap);
  }
  unsigned long long *hashed =  // tokens and documents hashed
      any_heldout ? reinterpret_cast<unsigned long long *>(rb2 + r2_hashed) : nullptr;
  if (any_heldout) {
    // per stream, see the kernel (zeroed with the control block)
    unsigned long long *frontier = reinterpret_cast<unsigned long long *>(zb + zb_front);
    unsigned long long *prog = reinterpret_cast<unsigned long long *>(zb + zb_prog);
    NS_CK(cudaEventRecord(side.t0, st));
    const uint32_t first_num = speculate ? 512u : 1024u;
    const int32_t *src = htok ? htok : c->tokens;
    int32_t *dst = htok ? c->tokens_rw : nullptr;
    // one launch over every stream, or one per copied group of streams
    const size_t n_groups = group_copy ? copy.done.size() : 1;
    for (size_t gi = 0; gi < n_groups; gi++) {
      const uint32_t j0 = group_copy ? copy.j_first[gi] : 0;
      const uint32_t j1 = group_copy ? copy.j_first[gi + 1] : J;
      if (group_copy) NS_CK(cudaStreamWaitEvent(st, copy.done[gi], 0));
      NS_CK(nsk::launch_hash_prefix(src, dst, tokens_read, hashed, c->offs, static_cast<uint32_t *>(d_sdb),
                                    static_cast<uint16_t *>(d_stream_bp), J, D0, order, klen,
                                    c->cum + (size_t)K * J, ready, S, T, c->G, c->hash_key,
                                    heldout_mode ? 1u : 0u, frontier, prog, j0, j1 - j0, nullptr,
                                    first_num, pre_cap, c->n_sms, st));
    }
    if (speculate) {
      // the fill needs the quota table; the second round every token
      if (group_copy) NS_CK(cudaStreamWaitEvent(st, copy.done.back(), 0));
      NS_CK(cudaStreamWaitEvent(st, side.join, 0));
      NS_CK(nsk::launch_fill_need(static_cast<uint32_t *>(d_sdb), J, D0,
                                  static_cast<uint16_t *>(d_stream_bp), order, klen, c->offs,
                                  c->n_tokens, c->cum + (size_t)K * J, T, c->G, first_num,
                                  pre_cap, need_num, st));
      NS_CK(nsk::launch_hash_prefix(src, dst, tokens_read, hashed, c->offs, static_cast<uint32_t *>(d_sdb),
                                    static_cast<uint16_t *>(d_stream_bp), J, D0, order, klen,
                                    c->cum + (size_t)K * J, ready, S, T, c->G, c->hash_key,
                                    heldout_mode ? 1u : 0u, frontier, prog, 0, J, need_num, 0,
                                    nullptr, c->n_sms, st));
    }
    NS_CK(cudaEventRecord(side.t1, st));
  }
  // every token is on the device before anything after the hash reads it
  if (group_copy) NS_CK(cudaStreamWaitEvent(st, copy.done.back(), 0));
  // greedy packing cuts documents into T-chunks; wrap packing keeps each
  // kept document whole as one piece (no document reaches 2^31 tokens)
  const uint32_t chunk = wrap ? 0x80000000u : T;
  NS_CK(nsk::launch_scan_pieces(klen, n_pos, chunk, kex, pex, scan_scratch, scan_bytes,
                                static_cast<uint32_t *>(d_sdb), J, D0, pos_lim, done_scan,
                                c->n_sms, st));
  // the cutoff reads the quota table, and the readback after it the error
  // word the offsets check sets: the side streams join here, after the scans
  NS_CK(cudaStreamWaitEvent(st, side.join, 0));
  NS_CK(cudaStreamWaitEvent(st, side.join2, 0));

  // ---- 4. the prefix of each stream the horizon reaches -------------------
  uint32_t *cutoff = reinterpret_cast<uint32_t *>(rb1);
  int64_t *npieces = reinterpret_cast<int64_t *>(rb1 + r1_np);
  int64_t *ptokens = reinterpret_cast<int64_t *>(rb1 + r1_pt);
  int64_t *node_base = reinterpret_cast<int64_t *>(rb1 + r1_nb);
  NS_CK(nsk::launch_cutoff(static_cast<uint32_t *>(d_sdb), J, D0, kex, pex, c->cum + (size_t)K * J,
                           T, c->G, need_num, pos_lim, cutoff, npieces, ptokens, node_base,
                           reinterpret_cast<uint32_t *>(rb1), (uint32_t)(r1_rmax / 4),
                           (uint32_t)(r1_err / 4), c->err, done_cutoff, st));
  char *h1 = static_cast<char *>(a.host(r1_bytes));
  NS_CK(cudaMemcpyAsync(h1, rb1, r1_bytes, cudaMemcpyDeviceToHost, st));
  NS_CK(cudaStreamSynchronize(st));
  const uint32_t *cut_h = reinterpret_cast<const uint32_t *>(h1);
  const int64_t *np_h = reinterpret_cast<const int64_t *>(h1 + r1_np);
  const int64_t *nb_h = reinterpret_cast<const int64_t *>(h1 + r1_nb);
  const int64_t *pt_h = reinterpret_cast<const int64_t *>(h1 + r1_pt);
  const int32_t *rmax32 = reinterpret_cast<const int32_t *>(h1 + r1_rmax);
  const uint16_t *num_h = reinterpret_cast<const uint16_t *>(h1 + r1_num);
  const uint32_t *lim_h = reinterpret_cast<const uint32_t *>(h1 + r1_lim);
  int err_host = 0;
  std::memcpy(&err_host, h1 + r1_err, sizeof(int));
  if (err_host == nsk::kDevBadOffsets) return NS_ERR_BAD_INPUT;
  if (err_host != 0) return NS_ERR_DEVICE;
  // a stream shuffled only in part whose windows need more than that part
  // holds: its cutoff runs to the stream's end
  if (pos_lim)
    for (uint32_t j = 0; j < J; j++)
      if (lim_h[j] < N[j] && cut_h[j] > lim_h[j]) return kRetryFullBound;
  std::vector<uint64_t> rmax(J);
  std::vector<int64_t> wbase(J + 1, 0);
  for (uint32_t j = 0; j < J; j++) {
    // windows the horizon can read: whole segments when they are shuffled
    rmax[j] = c->G ? ((uint64_t)rmax32[j] + c->G - 1) / c->G * c->G : (uint64_t)rmax32[j];
    wbase[j + 1] = wbase[j] + (int64_t)rmax[j];
  }
  const int64_t n_nodes = nb_h[J];
  if (n_nodes >= (int64_t)0x7FFFFFFF) return NS_ERR_INVALID_ARG;
  c->n_pieces = (uint64_t)(n_nodes - J);
  c->complete.resize(J);
  // Pointer-jumping levels: enough for any stream's window count.  A window
  // holds at least one piece, and two consecutive greedy windows hold more
  // than T tokens (the second one's first piece did not fit in the first),
  // so a prefix of p kept tokens packs fewer than 2 ceil(p / T) + 2 windows.
  int64_t max_windows = 0;
  for (uint32_t j = 0; j < J; j++) {
    c->complete[j] = (cut_h[j] == N[j]) ? 1 : 0;
    const int64_t by_tokens = 2 * ((pt_h[j] + (int64_t)T - 1) / (int64_t)T) + 1;
    max_windows = std::max(max_windows, std::min(np_h[j], by_tokens));
  }
  uint32_t L = 1;
  while ((1ll << L) < max_windows + 1) L++;
  if (wrap) L = 0;  // wrap windows are found by position, without pointer jumping
  c->levels = L;

  // One upload for what follows, kept with the context: each stream's first
  // window number and the block layouts of the piece expansion, the next
  // window search and the window starts.  The arrays of the phase (the piece
  // tables, the jump levels, the windows, the row table) are reserved in one
  // allocation of each kind.
  const int64_t n_win = std::max<int64_t>(wbase[J], 1);
  std::vector<uint32_t> expand_bb, next_bb, win_bb;
  void *d_wbase, *d_expand_bb, *d_next_bb = nullptr, *d_win_bb;
  {
    Staging up2;
    up2.add(wbase.data(), (J + 1) * sizeof(int64_t), &d_wbase);
    std::vector<uint64_t> cnt(J);
    for (uint32_t j = 0; j < J; j++) cnt[j] = std::max<uint64_t>(cut_h[j], 1);
    expand_bb = seg_layout(cnt, 256);
    up2.add(expand_bb.data(), expand_bb.size() * 4, &d_expand_bb);
    if (!wrap) {
      for (uint32_t j = 0; j < J; j++) cnt[j] = (uint64_t)np_h[j] + 1;
      next_bb = seg_layout(cnt, 256);
      up2.add(next_bb.data(), next_bb.size() * 4, &d_next_bb);
    }
    win_bb = seg_layout(rmax, 256);
    up2.add(win_bb.data(), win_bb.size() * 4, &d_win_bb);
    const auto R = Arena::rounded;
    const size_t nn = (size_t)n_nodes;
    const size_t keep = R(up2.host.size()) + 2 * R(nn * 8) + 2 * R(nn * 4) + R((size_t)J * 4) +
                        R((size_t)K * c->B * sizeof(int4));
    const size_t temp = (wrap ? 3 * R((size_t)n_win * 4) : R((size_t)L * nn * 4) +
                                                              R((size_t)n_win * 4)) +
                        R(((size_t)J + 1) * 8) + R(((size_t)J + 1) * 4);
    if (!a.reserve(keep, true) || !a.reserve(temp, false)) return NS_ERR_OOM;
    if ((rc = up2.commit(a, st, true))) return rc;
  }
  c->wbase = static_cast<int64_t *>(d_wbase);

  // ---- 5. tokens of the prefixes the hash did not read --------------------
  // (host tokens read in place only): on the second stream, beside the
  // piece tables, which do not read tokens; joined before the summary.  A
  // prefix holding more than three quarters of its stream's tokens is copied
  // whole by the copy engine (one contiguous run, the host link's fastest
  // path); the others by chunks of their kept tokens.
  bool prefix_copy = false;
  if (htok) {
    std::vector<uint64_t> ob;
    const bool bounds = stream_token_bounds(cfg, J, c->n_tokens, ob);
    const uint64_t chunk = nsk::copy_chunk_tokens();
    std::vector<uint64_t> cnt(J, 0);
    std::vector<std::pair<uint64_t, uint64_t>> whole;  // token ranges [begin, end)
    for (uint32_t j = 0; j < J; j++) {
      if (stream_bp[j] != 0 || pt_h[j] <= 0) continue;
      if (bounds && 4 * (uint64_t)pt_h[j] > 3 * (ob[j + 1] - ob[j])) {
        if (!whole.empty() && whole.back().second == ob[j])
          whole.back().second = ob[j + 1];
        else
          whole.emplace_back(ob[j], ob[j + 1]);
      } else {
        cnt[j] = ((uint64_t)pt_h[j] + chunk - 1) / chunk;
      }
    }
    std::vector<uint32_t> bb = seg_layout(cnt, 8);
    if (bb[J] > 0 || !whole.empty()) {
      NS_CK(cudaEventRecord(side.fork, st));
      NS_CK(cudaStreamWaitEvent(side.s, side.fork, 0));
      for (const auto &r : whole) {
        NS_CK(cudaMemcpyAsync(c->tokens_rw + r.first, cfg->tokens + r.first,
                              (r.second - r.first) * sizeof(int32_t), cudaMemcpyHostToDevice,
                              side.s));
        c->host_bytes += (r.second - r.first) * sizeof(int32_t);
      }
      if (bb[J] > 0) {
        void *d_bb;
        if ((rc = upload(a, bb.data(), bb.size() * 4, &d_bb, st))) return rc;
        nsk::SegGrid g{static_cast<uint32_t *>(d_bb), J, bb[J]};
        // the grid table is uploaded on the main stream: fork after it
        NS_CK(cudaEventRecord(side.fork, st));
        NS_CK(cudaStreamWaitEvent(side.s, side.fork, 0));
        NS_CK(nsk::launch_copy_prefix(g, static_cast<uint32_t *>(d_sdb), D0, cutoff,
                                      static_cast<uint16_t *>(d_stream_bp), order, klen, kex,
                                      c->offs, htok, c->tokens_rw, tokens_read, side.s));
      }
      NS_CK(cudaEventRecord(side.join, side.s));
      prefix_copy = true;
    }
  }

  // ---- 6. pieces, next window start, pointer jumping ----------------------
  c->node_src = a.keep<int64_t>(n_nodes);
  c->node_S = a.keep<int64_t>(n_nodes);
  c->node_doc = a.keep<int32_t>(n_nodes);
  c->node_mthr = a.keep<int32_t>(n_nodes);
  int32_t *levels = wrap ? nullptr : a.temp<int32_t>((size_t)L * n_nodes);
  NS_ALLOC(c->node_src);
  NS_ALLOC(c->node_S);
  NS_ALLOC(c->node_doc);
  NS_ALLOC(c->node_mthr);
  if (!wrap) NS_ALLOC(levels);
  {
    nsk::SegGrid g{static_cast<uint32_t *>(d_expand_bb), J, expand_bb[J]};
    NS_CK(nsk::launch_expand(g, static_cast<uint32_t *>(d_sdb), D0, cutoff, order, klen, kex, pex,
                             node_base, npieces, c->offs, c->loss_start, chunk, c->node_src,
                             c->node_doc, c->node_mthr, c->node_S, st));
  }
  if (!wrap) {
    nsk::SegGrid g{static_cast<uint32_t *>(d_next_bb), J, next_bb[J]};
    NS_CK(nsk::launch_next(g, node_base, npieces, c->node_S, T, levels, st));
  }
  // two levels per launch while two remain
  for (uint32_t l = 1; l < L;) {
    const int32_t *prev = levels + (size_t)(l - 1) * n_nodes;
    if (l + 1 < L) {
      NS_CK(nsk::launch_jump_two_levels(prev, n_nodes, levels + (size_t)l * n_nodes,
                                        levels + (size_t)(l + 1) * n_nodes, st));
      l += 2;
    } else {
      NS_CK(nsk::launch_jump_level(prev, n_nodes, levels + (size_t)l * n_nodes, st));
      l += 1;
    }
  }

  // ---- 7. windows: count, starts, the valid horizon ------------------------
  c->W = a.keep<uint32_t>(J);
  int32_t *win_start = a.temp<int32_t>(n_win);
  int32_t *win_end = wrap ? a.temp<int32_t>(n_win) : nullptr;
  int32_t *win_clip = wrap ? a.temp<int32_t>(n_win) : nullptr;
  c->row_win = a.keep<int4>((size_t)K * c->B);
  uint32_t *bad_inv = reinterpret_cast<uint32_t *>(rb2 + r2_bad);
  uint32_t *valid = reinterpret_cast<uint32_t *>(rb2 + r2_valid);
  NS_ALLOC(c->W);
  NS_ALLOC(win_start);
  if (wrap) {
    NS_ALLOC(win_end);
    NS_ALLOC(win_clip);
  }
  NS_ALLOC(c->row_win);
  nsk::SegGrid wg{static_cast<uint32_t *>(d_win_bb), J, win_bb[J]};
  if (wrap) {
    NS_CK(nsk::launch_wrap_windows(wg, node_base, npieces, c->node_S, cutoff,
                                   static_cast<uint32_t *>(d_sdb), J, T, c->W, c->wbase,
                                   win_start, win_end, win_clip, st));
  } else {
    NS_CK(nsk::launch_count_windows(levels, n_nodes, L, node_base, npieces, J, c->W, st));
    NS_CK(nsk::launch_window_starts(wg, levels, n_nodes, L, node_base, c->W, c->wbase,
                                    win_start, st));
  }
  // the row table; in the same launch, the valid horizon and each stream's
  // first item in the digest
  int64_t *ubase = a.temp<int64_t>(J + 1);
  NS_ALLOC(ubase);
  NS_CK(nsk::launch_row_table(c->rb, c->cum, c->W, c->wbase, win_start, levels, win_end, win_clip,
                              J, c->B, K, c->seed, c->G,
                              (c->flags & NS_PACK_SHUFFLE_ROWS) ? 1u : 0u, c->row_win, c->err,
                              bad_inv, (c->flags & NS_PACK_DRAIN) ? 1u : 0u, valid, ubase,
                              done_rows, st));

  // ---- 8. order digest, and the summary the host reads back ---------------
  unsigned long long *dacc = reinterpret_cast<unsigned long long *>(rb2 + r2_dacc);
  uint64_t *digest = reinterpret_cast<uint64_t *>(rb2 + r2_digest);
  nsk::DigestHeader h{};
  h.scalars[0] = T;
  h.scalars[1] = c->B;
  h.scalars[2] = K;
  h.scalars[3] = 0;  // valid_steps, read on the device
  h.scalars[4] = c->flags & (NS_PACK_DRAIN | NS_PACK_HELDOUT | NS_PACK_SHUFFLE_ROWS | NS_PACK_WRAP);
  h.scalars[5] = (uint64_t)(uint32_t)c->pad_id;
  h.scalars[6] = c->seed;
  h.scalars[7] = c->hash_key;
  h.scalars[8] = S;
  h.scalars[9] = J;
  h.scalars[10] = c->G;
  h.scalars[11] = c->len_bucket;
  h.source_weight = static_cast<uint32_t *>(d_sw);
  h.source_bp = static_cast<uint16_t *>(d_sbp);
  h.sdb = static_cast<uint32_t *>(d_sdb);
  h.ssrc = static_cast<uint32_t *>(d_ssrc);
  h.tw = static_cast<uint32_t *>(d_tw);
  h.piece_items = static_cast<uint64_t *>(d_piece_items);
  h.n_piece_items = piece_items.size();
  h.S = S;
  h.J = J;
  NS_CK(nsk::launch_digest(h, c->quota, K, wg, c->wbase, win_start, c->node_src, c->node_doc,
                           c->offs, valid, ubase, c->W, c->seed, c->G, win_clip, c->err, dacc,
                           digest, reinterpret_cast<uint32_t *>(rb2), (uint32_t)(r2_W / 4),
                           (uint32_t)(r2_err / 4), done_digest, st));

  // ---- 9. read back the summary ------------------------------------------
  // (the prefix copy, if any, adds its count of the tokens it read)
  if (prefix_copy) NS_CK(cudaStreamWaitEvent(st, side.join, 0));
  char *h2 = static_cast<char *>(a.host(r2_bytes));
  NS_CK(cudaMemcpyAsync(h2, rb2, r2_bytes, cudaMemcpyDeviceToHost, st));
  NS_CK(cudaStreamSynchronize(st));
  unsigned long long read_h = 0, hashed_h[2] = {0, 0};
  uint32_t valid_h = 0;
  uint64_t digest_h = 0;
  if (tokens_read) std::memcpy(&read_h, h2 + r2_read, 8);
  if (hashed) std::memcpy(hashed_h, h2 + r2_hashed, 16);
  std::memcpy(&digest_h, h2 + r2_digest, 8);
  std::memcpy(&valid_h, h2 + r2_valid, 4);
  std::memcpy(&err_host, h2 + r2_err, 4);
  const uint32_t *W_h = reinterpret_cast<const uint32_t *>(h2 + r2_W);
  if (err_host != 0) return NS_ERR_DEVICE;
  c->host_bytes += (uint64_t)read_h * sizeof(int32_t);
  c->hashed_tokens += hashed_h[0];
  c->hashed_docs += hashed_h[1];
  if (any_heldout) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, side.t0, side.t1) == cudaSuccess)
      c->hash_ns += (uint64_t)((double)ms * 1e6);
    cudaGetLastError();
  }
  // a stream cut short at a speculated bound must hold one window past the
  // ones the horizon reads (so that those are closed): else, the full bound
  for (uint32_t j = 0; j < J; j++)
    if (need_num && num_h[j] < 1024 && cut_h[j] < N[j] && (uint64_t)W_h[j] < rmax[j] + 1)
      return kRetryFullBound;
  c->windows.assign(W_h, W_h + J);
  c->valid_steps = valid_h;
  c->digest = digest_h;
  return NS_OK;
}

// A context with the recipe's scalars and no tables yet.
ns_pack_ctx *new_context(const ns_pack_config *cfg) {
  ns_pack_ctx *c = new (std::nothrow) ns_pack_ctx();
  if (!c) return nullptr;
  c->T = cfg->T;
  c->B = cfg->B;
  c->K = cfg->max_steps;
  c->flags = cfg->flags;
  c->G = cfg->window_segment;
  c->len_bucket = cfg->len_bucket;
  c->S = cfg->n_sources;
  c->J = cfg->n_streams;
  c->n_docs = cfg->n_docs;
  c->pad_id = cfg->pad_id;
  c->seed = cfg->seed;
  c->hash_key = cfg->hash_key;
  c->n_tokens = cfg->n_tokens;
  c->tokens = cfg->tokens;
  c->offs = cfg->doc_offsets;
  c->loss_start = cfg->loss_start;
  c->stream = static_cast<cudaStream_t>(cfg->cuda_stream);
  c->alloc = cfg->alloc;
  c->free_fn = cfg->free;
  c->user = cfg->alloc_user;
  return c;
}

}  // namespace

extern "C" {

int ns_pack_init(const ns_pack_config *cfg, ns_pack_ctx **out) {
  if (!out) return NS_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = check_config(cfg);
  if (rc) return rc;
  const uint64_t launches0 = nsk::launch_counter();
  uint64_t host_bytes_before = 0;  // a host corpus read by an earlier pass
  uint64_t hashed_before[3] = {0, 0, 0};  // tokens and documents it hashed, its time
  // pass 1 hashes to a speculated bound; pass 2, only if that left a stream
  // short of its windows, to the full bound
  for (uint32_t pass = 1; pass <= 2; pass++) {
    ns_pack_ctx *c = new_context(cfg);
    if (!c) return NS_ERR_OOM;
    c->speculate = (pass == 1);
    c->init_passes = pass;
    Arena a(c);
    rc = build(c, cfg, a);
    c->init_launches = (uint32_t)(nsk::launch_counter() - launches0);
    c->host_bytes += host_bytes_before;
    c->hashed_tokens += hashed_before[0];
    c->hashed_docs += hashed_before[1];
    c->hash_ns += hashed_before[2];
    if (rc == NS_OK) {
      a.release();
      *out = c;
      return NS_OK;
    }
    host_bytes_before = c->host_bytes;
    hashed_before[0] = c->hashed_tokens;
    hashed_before[1] = c->hashed_docs;
    hashed_before[2] = c->hash_ns;
    cudaStreamSynchronize(c->stream);
    cudaGetLastError();
    a.release();
    release_ctx(c);
    if (rc != kRetryFullBound) return rc;
  }
  return NS_ERR_DEVICE;  // the full bound cannot fall short
}

int ns_pack_step(ns_pack_ctx *ctx, uint32_t step0, uint32_t n_steps, uint32_t row_begin,
                 uint32_t row_end, const ns_pack_out *out, void *cuda_stream) {
  if (!ctx || !out || n_steps == 0) return NS_ERR_INVALID_ARG;
  if (row_begin >= row_end || row_end > ctx->B) return NS_ERR_INVALID_ARG;
  if (!out->tokens || !out->pos || !out->doc || !out->mask || !out->row_fp || !out->row_learned)
    return NS_ERR_INVALID_ARG;
  if ((uint64_t)step0 + n_steps <= ctx->K && ctx->piece_begin.size() > 1)
    for (uint32_t k = step0; k < step0 + n_steps; k++)
      if (row_end > rows_of_step(ctx, k)) return NS_ERR_INVALID_ARG;
  const uintptr_t al = reinterpret_cast<uintptr_t>(out->tokens) |
                       reinterpret_cast<uintptr_t>(out->pos) |
                       reinterpret_cast<uintptr_t>(out->doc) | reinterpret_cast<uintptr_t>(out->mask);
  if (al % 16 != 0) return NS_ERR_INVALID_ARG;
  if (!aligned_for(out->row_fp) || !aligned_for(out->row_learned) || !aligned_for(out->row_len))
    return NS_ERR_INVALID_ARG;
  if ((uint64_t)n_steps * (row_end - row_begin) >= (1ull << 31)) return NS_ERR_INVALID_ARG;
  if ((uint64_t)step0 + n_steps > ctx->K) return NS_ERR_HORIZON;
  if ((uint64_t)step0 + n_steps > ctx->valid_steps) return NS_ERR_EXHAUSTED;
  nsk::GatherParams p{};
  p.tokens = ctx->tokens;
  p.row_win = ctx->row_win;
  p.node_S = ctx->node_S;
  p.node_src = ctx->node_src;
  p.node_doc = ctx->node_doc;
  p.node_mthr = ctx->node_mthr;
  p.err = ctx->err;
  p.B = ctx->B;
  p.T = ctx->T;
  p.step0 = step0;
  p.n_steps = n_steps;
  p.row0 = row_begin;
  p.n_rows = row_end - row_begin;
  p.pad_id = ctx->pad_id;
  p.tokens_out = out->tokens;
  p.pos_out = out->pos;
  p.doc_out = out->doc;
  p.mask_out = out->mask;
  p.row_fp = out->row_fp;
  p.row_learned = out->row_learned;
  p.row_len = out->row_len;
  p.len_bucket = ctx->len_bucket;
  p.pad_tail = ctx->pad_tail;
  cudaStream_t st = cuda_stream ? static_cast<cudaStream_t>(cuda_stream) : ctx->stream;
  if (st != ctx->stream) ctx->foreign.store(true, std::memory_order_relaxed);
  if (nsk::launch_gather(p, st) != cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
  return NS_OK;
}

int ns_pack_batch_fp(ns_pack_ctx *ctx, const uint64_t *row_fp_dev, uint32_t n_steps,
                     uint32_t n_rows, uint64_t *batch_fp_dev, void *cuda_stream) {
  if (!ctx || !row_fp_dev || !batch_fp_dev || n_steps == 0 || n_rows == 0 ||
      n_steps >= (1u << 31))
    return NS_ERR_INVALID_ARG;
  if (!aligned_for(row_fp_dev) || !aligned_for(batch_fp_dev)) return NS_ERR_INVALID_ARG;
  cudaStream_t st = cuda_stream ? static_cast<cudaStream_t>(cuda_stream) : ctx->stream;
  if (nsk::launch_batch_fp(row_fp_dev, n_steps, n_rows, batch_fp_dev, st) != cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
  return NS_OK;
}

int ns_pack_step_learned(ns_pack_ctx *ctx, const int32_t *row_learned_dev, uint32_t n_steps,
                         uint32_t n_rows, int64_t *learned_dev, void *cuda_stream) {
  if (!ctx || !row_learned_dev || !learned_dev || n_steps == 0 || n_rows == 0 ||
      n_steps >= (1u << 31))
    return NS_ERR_INVALID_ARG;
  if (!aligned_for(row_learned_dev) || !aligned_for(learned_dev)) return NS_ERR_INVALID_ARG;
  cudaStream_t st = cuda_stream ? static_cast<cudaStream_t>(cuda_stream) : ctx->stream;
  if (nsk::launch_step_learned(row_learned_dev, n_steps, n_rows, learned_dev, st) !=
      cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
  return NS_OK;
}

static int read_error_word(ns_pack_ctx *ctx, cudaStream_t st) {
  int e = 0;
  if (cudaMemcpyAsync(&e, ctx->err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
  if (e == 0) return NS_OK;
  return e == nsk::kDevBadOffsets ? NS_ERR_BAD_INPUT : NS_ERR_DEVICE;
}

int ns_pack_fingerprint(ns_pack_ctx *ctx, const uint64_t *row_fp_dev, uint32_t n_rows,
                        uint64_t *batch_fp_host, void *cuda_stream) {
  if (!ctx || !row_fp_dev || !batch_fp_host || n_rows == 0) return NS_ERR_INVALID_ARG;
  if (!aligned_for(row_fp_dev)) return NS_ERR_INVALID_ARG;
  cudaStream_t st = cuda_stream ? static_cast<cudaStream_t>(cuda_stream) : ctx->stream;
  if (nsk::launch_batch_fp(row_fp_dev, 1, n_rows, ctx->fp_out, st) != cudaSuccess ||
      cudaMemcpyAsync(batch_fp_host, ctx->fp_out, sizeof(uint64_t), cudaMemcpyDeviceToHost, st) !=
          cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
  return read_error_word(ctx, st);
}

int ns_pack_info(const ns_pack_ctx *ctx, ns_pack_info_t *info) {
  if (!ctx || !info) return NS_ERR_INVALID_ARG;
  info->valid_steps = ctx->valid_steps;
  info->max_steps = ctx->K;
  info->n_streams = ctx->J;
  info->T = ctx->T;
  info->B = ctx->B;
  info->levels = ctx->levels;
  info->order_digest = ctx->digest;
  info->n_pieces = ctx->n_pieces;
  info->table_bytes = ctx->table_bytes;
  info->init_launches = ctx->init_launches;
  info->init_passes = ctx->init_passes;
  info->host_bytes = ctx->host_bytes;
  info->hashed_tokens = ctx->hashed_tokens;
  info->hashed_docs = ctx->hashed_docs;
  info->hash_ns = ctx->hash_ns;
  return NS_OK;
}

int ns_pack_stream_windows(const ns_pack_ctx *ctx, uint64_t *windows, uint8_t *complete) {
  if (!ctx) return NS_ERR_INVALID_ARG;
  if (windows) std::memcpy(windows, ctx->windows.data(), ctx->J * sizeof(uint64_t));
  if (complete) std::memcpy(complete, ctx->complete.data(), ctx->J);
  return NS_OK;
}

int ns_pack_quota_table(const ns_pack_ctx *ctx, int32_t *quota, int32_t *cum) {
  if (!ctx) return NS_ERR_INVALID_ARG;
  cudaStream_t st = ctx->stream;
  if (quota && cudaMemcpyAsync(quota, ctx->quota, (size_t)ctx->K * ctx->J * 4,
                               cudaMemcpyDeviceToHost, st) != cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
  if (cum && cudaMemcpyAsync(cum, ctx->cum, (size_t)(ctx->K + 1) * ctx->J * 4,
                             cudaMemcpyDeviceToHost, st) != cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
  return NS_OK;
}

int ns_pack_check(ns_pack_ctx *ctx) {
  if (!ctx) return NS_ERR_INVALID_ARG;
  return read_error_word(ctx, ctx->stream);
}

void ns_pack_free(ns_pack_ctx *ctx) {
  if (!ctx) return;
  if (ctx->foreign.load()) {
    // a step on another stream may still read the tables: wait for the device
    int cur = 0;
    if (cudaGetDevice(&cur) == cudaSuccess && cudaSetDevice(ctx->device) == cudaSuccess) {
      cudaDeviceSynchronize();
      cudaSetDevice(cur);
    }
  } else if (!(ctx->flags & NS_PACK_ORDERED_FREE) || !ctx->free_fn) {
    cudaStreamSynchronize(ctx->stream);
  }
  cudaGetLastError();
  release_ctx(ctx);
}

const char *ns_pack_strerror(int code) {
  switch (code) {
    case NS_OK: return "ok";
    case NS_ERR_INVALID_ARG: return "invalid argument";
    case NS_ERR_CUDA: return "CUDA runtime error";
    case NS_ERR_OOM: return "out of device memory";
    case NS_ERR_EXHAUSTED: return "a stream has no window left for this update";
    case NS_ERR_HORIZON: return "update index at or past max_steps";
    case NS_ERR_BAD_INPUT: return "doc_offsets malformed";
    case NS_ERR_DEVICE: return "a kernel recorded an inconsistency";
    default: return "unknown error";
  }
}

}  // extern "C"
