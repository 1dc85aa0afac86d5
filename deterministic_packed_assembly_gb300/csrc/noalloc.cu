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
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

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

}  // namespace

extern "C" int ns_pack_quota_noalloc(const uint32_t *source_weight, uint32_t n_sources,
                                     const uint32_t *stream_source, const uint32_t *stream_weight,
                                     uint32_t n_streams, uint32_t B, uint32_t max_steps,
                                     int32_t *quota_dev, int32_t *cum_dev, void *cuda_stream) {
  const uint32_t S = n_sources, J = n_streams, K = max_steps;
  if (!source_weight || !stream_source || !stream_weight || !quota_dev || !cum_dev)
    return NS_ERR_INVALID_ARG;
  if (S == 0 || S > NS_MAX_SOURCES || J == 0 || J > NS_MAX_STREAMS) return NS_ERR_INVALID_ARG;
  if (B == 0 || K == 0 || (uint64_t)K * B >= (1ull << 31)) return NS_ERR_INVALID_ARG;
  std::vector<uint32_t> src_first(S + 1, 0);
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
  // scratch layout: source weights | stream weights | source -> first stream
  // | the horizon as one piece (begin 0, B) | (beyond one warp) sources'
  // windows per update
  const size_t o_sw = 0;
  const size_t o_tw = o_sw + round256((size_t)S * 4);
  const size_t o_sf = o_tw + round256((size_t)J * 4);
  const size_t o_pc = o_sf + round256((size_t)(S + 1) * 4);  // one piece: begin 0, B
  const size_t o_sq = o_pc + 256;
  const size_t need = o_sq + (one_warp ? 0 : round256((size_t)K * S * 4));
  if (need > NS_NOALLOC_SCRATCH_BYTES) return NS_ERR_INVALID_ARG;

  unsigned char *scratch = nullptr;
  int rc = scratch_address(reinterpret_cast<void **>(&scratch));
  if (rc != NS_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  uint32_t *d_sw = reinterpret_cast<uint32_t *>(scratch + o_sw);
  uint32_t *d_tw = reinterpret_cast<uint32_t *>(scratch + o_tw);
  uint32_t *d_sf = reinterpret_cast<uint32_t *>(scratch + o_sf);
  uint32_t *d_pc = reinterpret_cast<uint32_t *>(scratch + o_pc);
  const uint32_t piece[2] = {0, B};
  if (cudaMemcpyAsync(d_sw, source_weight, (size_t)S * 4, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(d_tw, stream_weight, (size_t)J * 4, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(d_sf, src_first.data(), (size_t)(S + 1) * 4, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(d_pc, piece, sizeof(piece), cudaMemcpyHostToDevice, st) != cudaSuccess) {
    cudaGetLastError();
    return NS_ERR_CUDA;
  }
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
