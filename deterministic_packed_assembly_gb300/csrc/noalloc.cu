// ns_pack_quota_noalloc: the per-update quota tables of a recipe, computed
// without allocating any device memory.
//
// Who needs this: a caller that cannot call cudaMalloc.  A trainer that hands
// all of the GPU's memory to its own pool when it starts (so that its large
// allocations never fragment) has nothing left for a library to allocate
// outside that pool; a process that shares a GPU under a fixed memory budget
// may not grow past it; and cudaMalloc / cudaFree synchronise the device, which
// a caller in a tight loop cannot afford.  Such a caller passes its recipe (on
// the host) and two output buffers it already owns, and gets the same tables
// ns_pack_init builds and ns_pack_quota_table returns.
//
// Where the scratch lives: the kernels need the recipe's weight tables on the
// device and, for recipes beyond one warp (more than 32 sources or more than
// 32 strata in a source), a [max_steps][n_sources] table of the sources'
// windows per update.  Both go into one file-scope __device__ array of
// NS_NOALLOC_SCRATCH_BYTES, which every GPU that loads this library holds
// until the process exits.  Host code cannot use that array's name as a
// device address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it; make that
// first call before any stream capture.  Every call shares the one array:
// calls whose work overlaps on the GPU (different streams, or the same stream
// from several host threads without ordering) race on it.  Nothing in it has
// to start at zero: every byte a call reads is written earlier by that call.
//
// How the recipe reaches the device: a copy from pageable host memory may
// wait for the stream's earlier work, and the caller's arrays need not be
// page-locked.  So the weights travel in the parameter block of small upload
// kernels (a launch copies its parameters when it is enqueued): the call only
// enqueues kernels and returns without waiting on the stream.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "nspack.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[NS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return NS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return NS_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return NS_OK;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Words one upload launch carries.  A kernel's parameters may take up to
// 32,764 bytes on this architecture (CUDA 12.1 or later); 30 KB of words
// leaves room for the rest of the block.
constexpr uint32_t kUploadWords = 7680;
struct UploadBlock {
  uint32_t *dst;
  uint32_t n;
  uint32_t w[kUploadWords];
};
static_assert(sizeof(UploadBlock) <= 32000, "upload block beyond the parameter limit");

// dst[i] = w[i] for i < n.  __grid_constant__ lets the threads index the
// parameter block where it lies instead of each taking a private copy.
__global__ void __launch_bounds__(256) upload_words_kernel(const __grid_constant__ UploadBlock b) {
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < b.n; i += gridDim.x * blockDim.x)
    b.dst[i] = b.w[i];
}

// Per host thread, so that calls from several threads do not share them (the
// device scratch is shared regardless); fixed size, nothing allocated.
thread_local UploadBlock tl_block;
thread_local uint32_t tl_src_first[NS_MAX_SOURCES + 1];

}  // namespace

extern "C" int ns_pack_quota_noalloc(const uint32_t *source_weight, uint32_t n_sources,
                                     const uint32_t *stream_source, const uint32_t *stream_weight,
                                     uint32_t n_streams, uint32_t B, uint32_t max_steps,
                                     int32_t *quota_dev, int32_t *cum_dev, void *cuda_stream) {
  const uint32_t S = n_sources, J = n_streams, K = max_steps;
  if (!source_weight || !stream_source || !stream_weight || !quota_dev || !cum_dev)
    return NS_ERR_INVALID_ARG;
  // int32 tables: the kernels' 4-byte stores would fault on a misaligned one
  if (reinterpret_cast<uintptr_t>(quota_dev) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(cum_dev) % 4 != 0)
    return NS_ERR_INVALID_ARG;
  if (S == 0 || S > NS_MAX_SOURCES || J == 0 || J > NS_MAX_STREAMS) return NS_ERR_INVALID_ARG;
  if (B == 0 || K == 0 || (uint64_t)K * B >= (1ull << 31)) return NS_ERR_INVALID_ARG;
  uint32_t *src_first = tl_src_first;
  uint32_t max_strata = 0;
  for (uint32_t s = 0; s < S; s++)
    if (source_weight[s] == 0) return NS_ERR_INVALID_ARG;
  for (uint32_t j = 0; j < J; j++) {
    if (stream_weight[j] == 0 || stream_source[j] >= S) return NS_ERR_INVALID_ARG;
    if (j > 0 && stream_source[j] < stream_source[j - 1]) return NS_ERR_INVALID_ARG;
  }
  for (uint32_t s = 0, j = 0; s < S; s++) {
    src_first[s] = j;
    while (j < J && stream_source[j] == s) j++;
    src_first[s + 1] = j;
    const uint32_t n = src_first[s + 1] - src_first[s];
    if (n == 0 || n > NS_MAX_STRATA_PER_SOURCE) return NS_ERR_INVALID_ARG;
    if (n > max_strata) max_strata = n;
  }
  const bool one_warp = S <= 32 && max_strata <= 32;
  // scratch layout, in 32-bit words from the start: source weights [S] |
  // stream weights [J] | source -> first stream [S + 1] | the horizon as one
  // piece (begin 0, B); then, 256-byte aligned and only beyond one warp, the
  // sources' windows per update [K][S]
  const uint32_t w_sw = 0, w_tw = S, w_sf = S + J, w_pc = 2 * S + J + 1;
  const uint32_t n_words = w_pc + 2;
  const size_t o_sq = round256((size_t)n_words * 4);
  const size_t need = o_sq + (one_warp ? 0 : round256((size_t)K * S * 4));
  if (need > NS_NOALLOC_SCRATCH_BYTES) return NS_ERR_INVALID_ARG;

  unsigned char *scratch = nullptr;
  int rc = scratch_address(reinterpret_cast<void **>(&scratch));
  if (rc != NS_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  uint32_t *words = reinterpret_cast<uint32_t *>(scratch);
  // the words of the layout above, uploaded kUploadWords at a time
  auto word = [&](uint32_t i) -> uint32_t {
    if (i < w_tw) return source_weight[i - w_sw];
    if (i < w_sf) return stream_weight[i - w_tw];
    if (i < w_pc) return src_first[i - w_sf];
    return i == w_pc ? 0u : B;
  };
  UploadBlock &blk = tl_block;
  for (uint32_t i0 = 0; i0 < n_words; i0 += kUploadWords) {
    const uint32_t n = (n_words - i0 < kUploadWords) ? n_words - i0 : kUploadWords;
    blk.dst = words + i0;
    blk.n = n;
    for (uint32_t q = 0; q < n; q++) blk.w[q] = word(i0 + q);
    upload_words_kernel<<<(n + 255) / 256, 256, 0, st>>>(blk);
    ++nsk::launch_counter();
    if (cudaGetLastError() != cudaSuccess) return NS_ERR_CUDA;
  }
  const uint32_t *d_sw = words + w_sw;
  const uint32_t *d_tw = words + w_tw;
  const uint32_t *d_sf = words + w_sf;
  const uint32_t *d_pc = words + w_pc;
  const nsk::QuotaPieces qp{d_pc, d_pc + 1, d_sw, d_tw, 1};
  cudaError_t e;
  if (one_warp) {
    e = nsk::launch_quota_warp(qp, S, d_sf, J, K, max_strata, quota_dev, cum_dev, nullptr, st);
  } else {
    int32_t *d_sq = reinterpret_cast<int32_t *>(scratch + o_sq);
    e = nsk::launch_quota_sources(qp, S, K, d_sq, st);
    if (e == cudaSuccess)
      e = nsk::launch_quota_strata(qp, d_sq, d_sf, S, J, K, max_strata, quota_dev, cum_dev,
                                   nullptr, st);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
  return NS_OK;
}
