// ns_pack_probe_hash_terms: the held-out hash's per-token term in a loop
// that touches no memory -- the rate at which this GPU computes the terms
// with nothing else to do, which bounds the hash kernel from above (it is
// integer-bound: one SplitMix64 finaliser per token, two 64-bit multiplies
// and three 64-bit xor-shifts).  The term is the same device function the
// hash kernel calls; each thread feeds it in-document indices i0, i0 + 1, ...
// and tokens tok ^ t from registers (two integer operations a term that the
// hash kernel, whose tokens come from memory, spends on its own indices).
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "nspack_probe.h"

namespace {

constexpr uint32_t kProbeThreads = 256;

__global__ void __launch_bounds__(kProbeThreads)
    hash_terms_loop_kernel(uint32_t n, unsigned long long *__restrict__ sum) {
  const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t tok = tid * 2654435761u;
  const uint32_t i0 = tid & 1023u;
  uint64_t acc = 0;
#pragma unroll 8
  for (uint32_t t = 0; t < n; t++) acc += nsk::hash_term(i0 + t, tok ^ t);
  atomicAdd(sum, (unsigned long long)acc);
}

}  // namespace

extern "C" int ns_pack_probe_hash_terms(uint32_t blocks, uint32_t terms_per_thread,
                                        uint64_t *sum_dev, void *cuda_stream) {
  if (!sum_dev || blocks == 0 || blocks > (1u << 20)) return NS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(sum_dev) % 8 != 0) return NS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  hash_terms_loop_kernel<<<blocks, kProbeThreads, 0, st>>>(
      terms_per_thread, reinterpret_cast<unsigned long long *>(sum_dev));
  ++nsk::launch_counter();
  if (cudaGetLastError() != cudaSuccess) return NS_ERR_CUDA;
  return NS_OK;
}
