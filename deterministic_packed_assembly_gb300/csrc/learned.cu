// Learned positions of every update: the sum of its rows' learned counts,
// the count a trainer weighs the update's loss by (Linnet training docs,
// Supervised fine-tuning: a step's loss is normalised by its learned
// positions).  One block per update, a block-wide sum in 64 bits.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace nsk {
namespace {

__global__ void __launch_bounds__(256)
    step_learned_kernel(const int32_t *__restrict__ row_learned, uint32_t n_rows,
                        int64_t *__restrict__ out) {
  pdl_wait_then_release();
  __shared__ int64_t part[8];
  const int32_t *r = row_learned + (size_t)blockIdx.x * n_rows;
  int64_t acc = 0;
  for (uint32_t i = threadIdx.x; i < n_rows; i += blockDim.x) acc += __ldg(r + i);
  acc = warp_sum_i64(acc);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    int64_t v = (threadIdx.x < (blockDim.x >> 5)) ? part[threadIdx.x] : 0;
    v = warp_sum_i64(v);
    if (threadIdx.x == 0) out[blockIdx.x] = v;
  }
}

}  // namespace

cudaError_t launch_step_learned(const int32_t *row_learned, uint32_t n_steps, uint32_t n_rows,
                                int64_t *out, cudaStream_t st) {
  ++launch_counter();
  pdl_launch(step_learned_kernel, n_steps, 256, 0, st, row_learned, n_rows, out);
  return cudaGetLastError();
}

}  // namespace nsk
