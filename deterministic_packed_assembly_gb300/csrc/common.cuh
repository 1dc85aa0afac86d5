// Device helpers shared by the library's kernels (not by the CPU oracle).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace nsk {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

// Codes written into the context's device error word (first writer wins).
enum DevError : int {
  kDevOk = 0,
  kDevBadOffsets = 1,   // doc_offsets not a valid partition of the tokens
  kDevWindowTooLong = 2, // a window's pieces add up to more than T
  kDevWalkLimit = 3,    // Feistel cycle walk did not land in range (cannot happen)
  kDevBadNode = 4,      // a window start or piece index out of its table
};

// SplitMix64 finaliser as a pure function of x (Steele, Lea & Flood 2014).
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + kGolden;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// The held-out hash's term of the token `tok` at in-document index i.
__device__ __forceinline__ uint64_t hash_term(uint32_t i, uint32_t tok) {
  return splitmix64(((uint64_t)i << 32) | tok);
}

// Programmatic dependent launch: a kernel launched with it (pdl_launch) may
// be scheduled while the kernel before it in the stream drains.  It calls
// pdl_wait first thing: wait until that kernel has finished and its writes
// are visible (a no-op for a kernel launched the ordinary way).  Every
// kernel in a chain of such launches calls it before any early return, so
// that a grid never completes before the one it depends on.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// pdl_wait, then let the next kernel's blocks be scheduled at once (they
// wait in their own pdl_wait): for short kernels.  A long kernel with few
// blocks calls pdl_wait alone, else the next kernel's blocks would sit on
// the SMs, waiting, for all of its run.
__device__ __forceinline__ void pdl_wait_then_release() {
  pdl_wait();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `k` on `st` with programmatic dependent launch allowed: its blocks
// may be scheduled while the previous kernel in the stream drains, and wait
// in pdl_wait_then_release (which every such kernel calls first) for it to
// finish.  Errors go to cudaGetLastError, as with <<<...>>>.
template <typename... KArgs, typename... Args>
inline void pdl_launch(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ void set_error(int *word, int code) {
  if (word) atomicCAS(word, 0, code);
}

// Largest index i in [lo, hi) with a[i] <= x, for a nondecreasing; lo - 1
// when a[lo] > x.  Reads through the read-only path.
template <class T, class I>
__device__ __forceinline__ I last_le(const T *__restrict__ a, I lo, I hi, T x) {
  I l = lo, h = hi;  // invariant: answer in [l - 1, h - 1]
  while (l < h) {
    I m = l + (h - l) / 2;
    if (__ldg(a + m) <= x)
      l = m + 1;
    else
      h = m;
  }
  return l - 1;
}

// Same search over a table staged in shared memory.
template <class T, class I>
__device__ __forceinline__ I last_le_smem(const T *a, I lo, I hi, T x) {
  I l = lo, h = hi;
  while (l < h) {
    I m = l + (h - l) / 2;
    if (a[m] <= x)
      l = m + 1;
    else
      h = m;
  }
  return l - 1;
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int64_t warp_sum_i64(int64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int warp_sum_i32(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace nsk
