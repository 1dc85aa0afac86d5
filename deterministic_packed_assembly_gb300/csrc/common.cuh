// Device helpers shared by the library's kernels (not by the CPU oracle).
#pragma once

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
