// Kernels that build a packing context: offsets check, Feistel keys, the
// two-level quota tables, the held-out hash, the shuffled order, the scans of
// kept lengths and piece counts, piece expansion, next-window search, the
// pointer-jumping tables, window numbering, the valid-step horizon and the
// order digest.  All integer; every table is written once per context.
//
// What each step computes is stated in the NeuronSpark-Trainer README,
// Concepts (held-out split by a hash of the text; shuffled documents;
// per-update source and stratum shares; windows cut at document ends) and in
// the Linnet training docs, Supervised fine-tuning (rows of exactly T
// positions, padded).
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace nsk {

namespace {

constexpr int kThreads = 256;
// The held-out hash: 128-thread CTAs, 7 per SM (72 registers a thread, no
// spills; its warps are independent, so only the count per SM matters).
constexpr int kHashThreads = 128;
constexpr int kHashBlocksPerSM = 7;
// 16-byte blocks a lane loads per step of the hash (128 tokens each), and as
// many more in flight for the next step
constexpr uint32_t kHashBlocksPerLane = 4;

inline unsigned blocks_for(uint64_t n, int threads = kThreads) {
  return (unsigned)((n + threads - 1) / threads);
}

// Stream j of block b of a segmented launch, and the block's index within
// the stream's run of blocks.
__device__ __forceinline__ void seg_locate_at(const SegGrid &g, uint32_t b, uint32_t &j,
                                              uint32_t &blk) {
  __shared__ uint32_t s_j;
  if (threadIdx.x == 0) {
    int64_t jj = last_le<uint32_t, int64_t>(g.blk_base, 0, (int64_t)g.J, b);
    s_j = (uint32_t)(jj < 0 ? 0 : jj);
  }
  __syncthreads();
  j = s_j;
  blk = b - g.blk_base[j];
}
__device__ __forceinline__ void seg_locate(const SegGrid &g, uint32_t &j, uint32_t &blk) {
  seg_locate_at(g, blockIdx.x, j, blk);
}

// Every thread of the block calls it once its writes are done: true, in
// every thread of the block, for the last block of the grid to get here
// (*done counts the blocks, zeroed before the launch).  Each block's writes
// are made visible before it counts itself, so the last one reads every
// other block's results (through loads that do not take a line cached
// before, e.g. __ldcg).  No block waits for another.
__device__ __forceinline__ bool last_block_done(unsigned *done) {
  __shared__ bool s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (s_last) __threadfence();
  return s_last;
}

// Exclusive prefix of one value per thread over the block (blockDim.x a
// multiple of 32); *total gets the block's sum in every thread.  ws: 33
// words of shared memory, free again when it returns.
__device__ __forceinline__ int64_t block_excl_scan(int64_t v, int64_t *ws, int64_t *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[w] = x;
  __syncthreads();
  if (w == 0) {
    int64_t t = (lane < nw) ? ws[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    ws[lane] = t;
  }
  __syncthreads();
  const int64_t excl = (w ? ws[w - 1] : 0) + x - v;
  *total = ws[nw - 1];
  __syncthreads();
  return excl;
}

template <class T>
__device__ T block_sum(T v, T *scratch /* [33] */) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) scratch[w] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int nw = (blockDim.x + 31) >> 5;
    T t = (l < nw) ? scratch[l] : T(0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (l == 0) scratch[32] = t;
  }
  __syncthreads();
  T r = scratch[32];
  __syncthreads();
  return r;
}

// Windows of a stream the horizon can read: its last quota count, rounded up
// to whole segments when windows are read in a shuffled order within them.
__device__ __forceinline__ int64_t windows_needed(int32_t rmax, uint32_t G) {
  return G ? ((int64_t)rmax + G - 1) / G * G : (int64_t)rmax;
}

// Kept tokens a stream's prefix must exceed: num / 1024 of its windows times
// T (num 1024: the bound that holds for any packing; smaller: a bound
// speculated from the stream's measured fill, checked after packing).
__device__ __forceinline__ int64_t tokens_needed(int32_t rmax, uint32_t G, uint32_t T,
                                                 uint32_t num) {
  // windows < 2^31 and T <= 2^24, so wt < 2^55: floor(wt * num / 1024) taken
  // in two parts so that no product leaves 64 bits
  const uint64_t wt = (uint64_t)windows_needed(rmax, G) * T;
  return (int64_t)((wt >> 10) * num + (((wt & 1023u) * num) >> 10));
}

// ---------------------------------------------------------------------------
// doc_offsets must start at >= 0, never decrease, keep every length below
// 2^31 and end inside the token array.
// Each warp checks runs of 128 consecutive offsets: lane l holds offsets
// run + 32q + l (q = 0..3, each load a contiguous 256 bytes), takes its
// neighbour from the next lane (or the next quarter's first lane, or one
// extra load at the run's end), and the grid strides over the runs.
constexpr uint32_t kValidateRun = 128;

__global__ void __launch_bounds__(kThreads)
    validate_offsets_kernel(const int64_t *__restrict__ offs, uint32_t n_docs,
                            uint64_t n_tokens, int *err) {
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x >> 5);
  bool bad = false;
  for (uint64_t run = (uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       run * kValidateRun <= n_docs; run += warps) {
    const uint64_t b = run * kValidateRun;
    int64_t v[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const uint64_t e = b + 32u * q + lane;
      v[q] = (e <= n_docs) ? __ldcs(offs + e) : 0;
    }
    const int64_t tail =
        (lane == 31 && b + kValidateRun <= n_docs) ? __ldcs(offs + b + kValidateRun) : 0;
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const int64_t down = __shfl_down_sync(0xffffffffu, v[q], 1);
      const int64_t wrap = __shfl_sync(0xffffffffu, q < 3 ? v[q < 3 ? q + 1 : 0] : 0, 0);
      const int64_t next = lane < 31 ? down : (q < 3 ? wrap : tail);
      const uint64_t e = b + 32u * q + lane;
      if (e < n_docs) {
        const int64_t len = next - v[q];
        bad |= len < 0 || len > 0x7FFFFFFF;
      }
      if (e == 0) bad |= v[q] < 0;
      if (e == n_docs) bad |= v[q] < 0 || (uint64_t)v[q] > n_tokens;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, kDevBadOffsets);
}

// Round keys of the shuffle: K_r = splitmix64(splitmix64(seed) ^
// splitmix64((stream << 8) | r)), r = 0..3; thread 4 j + r writes K_r of
// stream j.  With est_tok, thread 4 j also bounds the positions the shuffle
// takes of stream j (pos_lim[j]): a stream without a held-out rate needs
// only about the documents that hold its estimated tokens, a quarter over
// and 1024 more (offsets are checked by their own kernel); every position
// of the others.
__global__ void keys_bound_kernel(uint64_t seed, uint32_t J, uint64_t *keys,
                                  const uint32_t *__restrict__ sdb,
                                  const int64_t *__restrict__ offs,
                                  const uint16_t *__restrict__ stream_bp,
                                  const unsigned long long *__restrict__ est_tok,
                                  uint32_t *__restrict__ pos_lim) {
  pdl_wait_then_release();
  uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (uint64_t)J * 4) return;
  const uint64_t j = i >> 2, r = i & 3;
  keys[i] = splitmix64(splitmix64(seed) ^ splitmix64((j << 8) | r));
  if (!est_tok || r != 0) return;
  const uint32_t b = sdb[j], e = sdb[j + 1];
  const uint64_t N = e - b;
  uint64_t lim = N;
  if (stream_bp[j] == 0 && N > 0) {
    const int64_t tok = offs[e] - offs[b];
    if (tok > 0) {
      const double want = 1.25 * (double)est_tok[j] * (double)N / (double)tok + 1024.0;
      if (want < (double)N) lim = (uint64_t)want;
    }
  }
  pos_lim[j] = (uint32_t)lim;
}

// ---------------------------------------------------------------------------
// A block that has written its streams' last row of the quota table (the
// windows each stream gives the whole horizon) counts itself done, so a
// kernel running beside it can start using those rows once every block has.
__device__ __forceinline__ void publish_ready(unsigned *ready) {
  if (!ready) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ready, 1u);
  }
}

// One update of the apportionment among this block's children (thread c owns
// child c; inactive threads hold weight 0).  n units now, N counting every
// update so far including this one; C is the child's count before.
//   base_c = floor(n v_c / V); R = n - sum base;
//   delta_c = N v_c - V (C_c + base_c)  (exact, 128-bit);
//   the R children with the largest delta (ties: lower index) get one more.
// Children ranked by (shortfall desc, index asc); with more than
// kRankDirect of them a bitonic sort of (shortfall, index) over the block
// (blockDim.x a power of two) replaces counting each child's rank against
// all others, so an update costs O(n log^2 n) compare-exchanges, not O(n^2).
constexpr int kRankDirect = 64;

__device__ __forceinline__ int64_t apportion_one(bool act, uint64_t v, uint64_t V, int64_t n,
                                                 int64_t N, int64_t C, int n_children,
                                                 __int128 *delta, int *order_s, int64_t *scratch) {
  int64_t base = act ? (int64_t)(((uint64_t)n * v) / V) : 0;
  int64_t R = n - block_sum<int64_t>(base, scratch);
  __int128 d = 0;
  if (act) d = (__int128)N * (__int128)v - (__int128)V * (__int128)(C + base);
  const int c = threadIdx.x;
  int64_t a = base;
  if (n_children <= kRankDirect) {
    if (act) delta[c] = d;
    __syncthreads();
    if (act) {
      int rank = 0;
      for (int c2 = 0; c2 < n_children; c2++) {
        __int128 e = delta[c2];
        rank += (e > d) || (e == d && c2 < c);
      }
      a += (rank < R) ? 1 : 0;
    }
    __syncthreads();
    return a;
  }
  // sort: inactive slots carry the smallest shortfall, after every child
  const __int128 kLow = (__int128)1 << 127;  // the most negative value
  delta[c] = act ? d : kLow;
  order_s[c] = c;
  __syncthreads();
  const int P2 = (int)blockDim.x;
  for (int k = 2; k <= P2; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      const int ix = c ^ jj;
      if (ix > c) {
        const __int128 dc = delta[c], dx = delta[ix];
        const int oc = order_s[c], ox = order_s[ix];
        // does slot ix's child come before slot c's (larger shortfall, or
        // equal and lower index)?
        const bool x_first = dx > dc || (dx == dc && ox < oc);
        const bool swap = ((c & k) == 0) ? x_first : !x_first;
        if (swap) {
          delta[c] = dx;
          delta[ix] = dc;
          order_s[c] = ox;
          order_s[ix] = oc;
        }
      }
      __syncthreads();
    }
  }
  // slot r holds the child of rank r: the first R get one more
  const int child = order_s[c];
  __syncthreads();
  order_s[child] = (c < R) ? 1 : 0;
  __syncthreads();
  if (act) a += order_s[c];
  __syncthreads();
  return a;
}

// Source level: every update of piece p hands out B_p windows among the
// sources, with the piece's weights; the rule's counts start again at every
// piece.
__global__ void quota_sources_kernel(QuotaPieces q, uint32_t S, uint32_t K,
                                     int32_t *__restrict__ src_quota) {
  pdl_wait();
  __shared__ __int128 delta[1024];
  __shared__ int order_s[1024];
  __shared__ int64_t scratch[33];
  __shared__ uint64_t uscratch[33];
  const bool act = threadIdx.x < S;
  for (uint32_t p = 0; p < q.P; p++) {
    const uint32_t k0 = q.begin[p], k1 = (p + 1 < q.P) ? q.begin[p + 1] : K;
    const int64_t Bp = q.B[p];
    const uint64_t v = act ? q.sw[(size_t)p * S + threadIdx.x] : 0;
    const uint64_t V = block_sum<uint64_t>(v, uscratch);
    int64_t C = 0;
    for (uint32_t k = k0; k < k1; k++) {
      int64_t a = apportion_one(act, v, V, Bp, (int64_t)(k - k0 + 1) * Bp, C, (int)S, delta,
                                order_s, scratch);
      if (act) src_quota[(size_t)k * S + threadIdx.x] = (int32_t)a;
      C += a;
    }
  }
}

// Stratum level: block s splits source s's windows of every update among its
// streams; writes the per-stream quota and the windows each stream has given
// before each update (which run on across pieces).
__global__ void quota_strata_kernel(QuotaPieces q, const int32_t *__restrict__ src_quota,
                                    const uint32_t *__restrict__ src_first, uint32_t S,
                                    uint32_t J, uint32_t K, int32_t *__restrict__ quota,
                                    int32_t *__restrict__ cum, unsigned *ready) {
  pdl_wait();
  __shared__ __int128 delta[1024];
  __shared__ int order_s[1024];
  __shared__ int64_t scratch[33];
  __shared__ uint64_t uscratch[33];
  const uint32_t s = blockIdx.x;
  const uint32_t f0 = src_first[s], f1 = src_first[s + 1];
  const int n_st = (int)(f1 - f0);
  const bool act = (int)threadIdx.x < n_st;
  const uint32_t j = f0 + threadIdx.x;
  int64_t Cg = 0;
  for (uint32_t p = 0; p < q.P; p++) {
    const uint32_t k0 = q.begin[p], k1 = (p + 1 < q.P) ? q.begin[p + 1] : K;
    const uint64_t v = act ? q.tw[(size_t)p * J + j] : 0;
    const uint64_t V = block_sum<uint64_t>(v, uscratch);
    int64_t C = 0, Cs = 0;
    for (uint32_t k = k0; k < k1; k++) {
      const int64_t n = src_quota[(size_t)k * S + s];
      int64_t a = apportion_one(act, v, V, n, Cs + n, C, n_st, delta, order_s, scratch);
      if (act) {
        quota[(size_t)k * J + j] = (int32_t)a;
        cum[(size_t)k * J + j] = (int32_t)Cg;
      }
      C += a;
      Cg += a;
      Cs += n;
    }
  }
  if (act) cum[(size_t)K * J + j] = (int32_t)Cg;
  publish_ready(ready);
}

// Rank of this lane's value among lanes [0, count) by (value desc, lane asc);
// the value is a 128-bit integer split into a signed high and unsigned low
// half.  MAXC >= count bounds the fully unrolled loop, so the shuffles issue
// back to back; when every value fits in 64 bits (the usual case: a shortfall
// is a few windows times the weight sum) half the shuffles suffice.
template <int MAXC>
__device__ __forceinline__ int warp_rank128(int64_t hi, uint64_t lo, int count, int lane) {
  const bool fits = hi == ((int64_t)lo >> 63);
  int r = 0;
  if (__all_sync(0xffffffffu, fits || lane >= count)) {
    const int64_t x = (int64_t)lo;
#pragma unroll
    for (int j = 0; j < MAXC; j++) {
      const int64_t y = __shfl_sync(0xffffffffu, x, j);
      r += (j < count && (y > x || (y == x && j < lane))) ? 1 : 0;
    }
  } else {
#pragma unroll
    for (int j = 0; j < MAXC; j++) {
      const int64_t h = __shfl_sync(0xffffffffu, hi, j);
      const uint64_t l = __shfl_sync(0xffffffffu, lo, j);
      r += (j < count && (h > hi || (h == hi && (l > lo || (l == lo && j < lane))))) ? 1 : 0;
    }
  }
  return r;
}

// The same two-level rule as quota_sources_kernel + quota_strata_kernel for
// recipes with at most 32 sources and 32 strata per source: one warp per
// source replays the source level (identical in every block) and splits its
// source's windows among the strata.  The shortfalls are carried forward
// instead of recomputed: at the source level delta_c grows by B_p v_c - V a_c
// per update; at the stratum level D_c = Cs v_c - V_s C_c grows by
// n v_c - V_s a_c, and the source's n is its floor share or one more, so both
// floors of the strata are computed once per piece of the schedule (where
// every count starts again).  With a_c its floor share plus 0 or 1, each of
// those growths is the remainder of the floor division (below the weight
// sum, 64 bits) less the weight sum or nothing: the 128-bit shortfalls only
// ever add 64-bit numbers.
template <int SMAX, int TMAX>
__global__ void __launch_bounds__(32)
    quota_warp_kernel(QuotaPieces q, uint32_t S, const uint32_t *__restrict__ src_first,
                      uint32_t J, uint32_t K, int32_t *__restrict__ quota,
                      int32_t *__restrict__ cum, unsigned *ready) {
  pdl_wait();
  const int lane = threadIdx.x;
  const uint32_t s = blockIdx.x;
  const bool act = lane < (int)S;
  const uint32_t f0 = src_first[s];
  const int n_st = (int)(src_first[s + 1] - f0);
  const bool sact = lane < n_st;
  if (S == 1 && n_st == 1) {
    // one stream: the rule gives it every window of every update (floor
    // share n, no remainder), so the updates are written in parallel
    int64_t C0 = 0;  // windows given before the piece
    for (uint32_t p = 0; p < q.P; p++) {
      const uint32_t k0 = q.begin[p], k1 = (p + 1 < q.P) ? q.begin[p + 1] : K;
      const int64_t Bp = q.B[p];
      for (uint32_t k = k0 + lane; k < k1; k += 32) {
        quota[(size_t)k * J + f0] = (int32_t)Bp;
        cum[(size_t)k * J + f0] = (int32_t)(C0 + (int64_t)(k - k0) * Bp);
      }
      C0 += (int64_t)(k1 - k0) * Bp;
    }
    if (lane == 0) cum[(size_t)K * J + f0] = (int32_t)C0;
    publish_ready(ready);
    return;
  }
  int64_t Cg = 0;  // windows this lane's stream has given (runs on across pieces)
  for (uint32_t p = 0; p < q.P; p++) {
    const uint32_t k0 = q.begin[p], k1 = (p + 1 < q.P) ? q.begin[p + 1] : K;
    const uint64_t Bp = q.B[p];
    // source level
    const uint64_t v = act ? q.sw[(size_t)p * S + lane] : 0;
    const uint64_t V = warp_sum_u64(v);
    const int64_t base = act ? (int64_t)((Bp * v) / V) : 0;
    const int64_t R = (int64_t)Bp - warp_sum_i64(base);
    const int64_t rem = (int64_t)(Bp * v - V * (uint64_t)base);  // in [0, V)
    __int128 delta = rem;
    // stratum level of source s
    const uint64_t w = sact ? q.tw[(size_t)p * J + f0 + lane] : 0;
    const uint64_t Vs = warp_sum_u64(w);
    const int64_t bs = __shfl_sync(0xffffffffu, base, (int)s);
    const int64_t b0 = sact ? (int64_t)(((uint64_t)bs * w) / Vs) : 0;
    const int64_t b1 = sact ? (int64_t)(((uint64_t)(bs + 1) * w) / Vs) : 0;
    const int64_t R0 = bs - warp_sum_i64(b0);
    const int64_t R1 = bs + 1 - warp_sum_i64(b1);
    // n w - V_s * (floor share) for n = bs and n = bs + 1, each in [0, V_s)
    const int64_t r0 = (int64_t)((uint64_t)bs * w - Vs * (uint64_t)b0);
    const int64_t r1 = (int64_t)((uint64_t)(bs + 1) * w - Vs * (uint64_t)b1);
    __int128 D = 0;
    for (uint32_t k = k0; k < k1; k++) {
      const int rs = warp_rank128<SMAX>((int64_t)(delta >> 64), (uint64_t)delta, (int)S, lane);
      const bool extra = act && rs < R;
      const int64_t a = base + (extra ? 1 : 0);
      delta += (__int128)(extra ? rem - (int64_t)V : rem);
      const int64_t n = __shfl_sync(0xffffffffu, a, (int)s);
      if (TMAX == 1) {
        // one stratum: it takes all of its source's windows
        if (sact) {
          quota[(size_t)k * J + f0 + lane] = (int32_t)n;
          cum[(size_t)k * J + f0 + lane] = (int32_t)Cg;
        }
        Cg += n;
        continue;
      }
      const bool lo_share = (n == bs);
      const int64_t bsel = lo_share ? b0 : b1;
      const int64_t Rsel = lo_share ? R0 : R1;
      const __int128 d2 = D + (__int128)(lo_share ? r0 : r1);
      const int rt = warp_rank128<TMAX>((int64_t)(d2 >> 64), (uint64_t)d2, n_st, lane);
      const bool extra2 = sact && rt < Rsel;
      const int64_t a2 = bsel + (extra2 ? 1 : 0);
      if (sact) {
        quota[(size_t)k * J + f0 + lane] = (int32_t)a2;
        cum[(size_t)k * J + f0 + lane] = (int32_t)Cg;
      }
      Cg += a2;
      D = extra2 ? d2 - (__int128)(int64_t)Vs : d2;
    }
  }
  if (sact) cum[(size_t)K * J + f0 + lane] = (int32_t)Cg;
  publish_ready(ready);
}

// rb[k][j]: the first row of stream j in update k (rows ordered by stream).
// One block per update, a block-wide scan over the streams.
__global__ void __launch_bounds__(256)
    row_base_kernel(const int32_t *__restrict__ quota, uint32_t J, int32_t *__restrict__ rb) {
  pdl_wait_then_release();
  __shared__ int64_t ws[33];
  const uint32_t k = blockIdx.x;
  const int32_t *q = quota + (size_t)k * J;
  int32_t *r = rb + (size_t)k * (J + 1);
  int64_t carry = 0;
  for (uint32_t c0 = 0; c0 < J; c0 += blockDim.x) {
    const uint32_t j = c0 + threadIdx.x;
    int64_t total;
    const int64_t e = block_excl_scan((j < J) ? q[j] : 0, ws, &total);
    if (j < J) r[j] = (int32_t)(carry + e);
    carry += total;
  }
  if (threadIdx.x == 0) r[J] = (int32_t)carry;
}

// ---------------------------------------------------------------------------
// Held-out hash.  acc_d = sum_i splitmix64((i << 32) | u32 tok_i),
// h_d = splitmix64(acc_d ^ splitmix64(hash_key + L_d)); held out iff
// floor(h_d * 10000 / 2^64) < bp of the document's source.  One warp per
// document, reading aligned 16-byte blocks that each hold at least one of its
// tokens, four blocks per lane in flight (512 tokens per warp step).
//
// Four tokens that all lie inside the document, the first at in-document
// index i0 (documents are shorter than 2^31 tokens).
__device__ __forceinline__ uint64_t hash_terms_inside(int4 v, uint32_t i0) {
  return hash_term(i0, (uint32_t)v.x) + hash_term(i0 + 1, (uint32_t)v.y) +
         hash_term(i0 + 2, (uint32_t)v.z) + hash_term(i0 + 3, (uint32_t)v.w);
}

// Terms of a block whose first token has in-document index i0, taken modulo
// 2^32 (the head block of a document that does not start on a 16-byte
// boundary has i0 "below" zero); a token whose index is not in [0, L) adds
// nothing.  Every lane computes all four mixes and masks them, so a warp
// whose blocks straddle a document edge runs one path, not two.
__device__ __forceinline__ uint64_t hash_terms_masked(int4 v, uint32_t i0, uint32_t L) {
  const int32_t e[4] = {v.x, v.y, v.z, v.w};
  uint64_t s = 0;
#pragma unroll
  for (int q = 0; q < 4; q++) {
    const uint32_t i = i0 + (uint32_t)q;
    const uint64_t t = hash_term(i, (uint32_t)e[q]);
    s += (i < L) ? t : 0ull;
  }
  return s;
}

// The whole warp sums the token terms of tokens[o0, o0 + L); every lane gets
// the sum.  Offsets are taken relative to the 16-byte block holding the
// first token, in 32 bits (documents are shorter than 2^31 tokens).  With
// kCopy, every block read is also written to the same place in dst (a
// corpus read from host memory lands in the device copy as it is hashed;
// the few tokens of neighbouring documents that share the first and last
// blocks are written with the values they have).
template <bool kCopy>
__device__ __forceinline__ uint64_t warp_doc_terms(const int32_t *__restrict__ tokens,
                                                   int32_t *__restrict__ dst, int64_t o0,
                                                   uint32_t L, int lane) {
  constexpr uint32_t U = kHashBlocksPerLane, kStep = 128 * U;
  const int64_t a0 = o0 & ~(int64_t)3;
  const uint32_t sh = (uint32_t)(o0 - a0);
  const int4 *base = reinterpret_cast<const int4 *>(tokens + a0);
  int4 *dbase = kCopy ? reinterpret_cast<int4 *>(dst + a0) : nullptr;
  const uint32_t end = L + sh;
  const uint32_t l4 = 4 * (uint32_t)lane;
  uint64_t acc = 0;
  int4 v[U];
#pragma unroll
  for (int u = 0; u < (int)U; u++) {
    const uint32_t ru = l4 + 128 * u;
    v[u] = make_int4(0, 0, 0, 0);
    if (ru < end) v[u] = __ldcs(base + (ru >> 2));
  }
  // r0: the step's first block offset, the same in every lane
  for (uint32_t r0 = 0; r0 < end; r0 += kStep) {
    // the next step's loads go out before this step's terms
    int4 w[U];
#pragma unroll
    for (int u = 0; u < (int)U; u++) {
      const uint32_t ru = r0 + kStep + 128 * u + l4;
      w[u] = make_int4(0, 0, 0, 0);
      if (ru < end) w[u] = __ldcs(base + (ru >> 2));
    }
    // each group of 128 tokens (one block per lane) is decided for the whole
    // warp: inside the document -> no checks; across an edge -> masked terms
#pragma unroll
    for (int u = 0; u < (int)U; u++) {
      const uint32_t b0 = r0 + 128 * u;
      if (kCopy && b0 + l4 < end) dbase[(b0 >> 2) + lane] = v[u];
      if (b0 >= sh && b0 + 128 <= end)
        acc += hash_terms_inside(v[u], b0 + l4 - sh);
      else if (b0 < end)
        acc += hash_terms_masked(v[u], b0 + l4 - sh, L);
    }
#pragma unroll
    for (int u = 0; u < (int)U; u++) v[u] = w[u];
  }
  return warp_sum_u64(acc);
}

// Held-out flags for the prefix of every stream the horizon reaches.  A
// stream's documents are taken in shuffled-position order, a few at a time
// from the stream's frontier; a document the stream does not keep (held out
// for training, not held out for validation) has its kept length set to 0.
// A warp takes more of a stream while its progress word (below) stays at
// or under need_j = num_j / 1024 of rmax_j * T (rmax_j * T: the windows the
// horizon asks of it hold at most that many; num_j from need_num, or
// need_num_all for every stream), and goes on to the next stream once the
// word passes need_j or the stream runs out.  A second launch with a larger
// num_j carries on from the first's frontier and words.  Every position
// below the final frontier is hashed, and the kept tokens below it exceed
// need_j unless the whole stream was hashed, so the prefix the cutoff kernel
// then takes (with the same num_j) only ever holds decided documents.  Warps
// start on different streams so that few overshoot any one stream.
// With kCopy the tokens are read from host memory the device can address
// and every hashed document is written to copy_dst; tokens_read counts them.
//
// A stream's progress word: bits 16 and up hold the kept tokens of the
// documents already decided plus, for each grab in flight, an estimate of
// the tokens it will keep (grab_estimate); bits 0..15 count the grabs in
// flight (at most one a warp: fewer than 2^16).  Counting grabs in flight
// keeps the warps that pile onto the last streams of a round from each
// taking one more grab once the need is already in flight.  The estimate
// only sets how far past need_j a stream is hashed: a warp reads the word
// again after each grab it finishes, and after the last update that leaves
// no grab in flight the word holds the decided kept tokens exactly, so the
// warp that made it takes more if they do not exceed need_j.  One word, so
// that both parts are read and updated together.  (A stream holds fewer
// than 2^47 tokens: the corpus is copied to the device whole.)
//
// The estimate: the expected kept fraction less 1/8 of the grab's tokens,
// which its documents keep almost surely (when they do not, the warp that
// decides the last of them takes the rest one grab at a time).  A stream
// that keeps at most 1/8 of its tokens (the validation stream) estimates
// nothing: its word is then its decided kept tokens alone, and its grabs are
// not counted either.
__device__ __forceinline__ uint32_t grab_share(uint32_t bp, uint32_t want_heldout) {
  const uint32_t keep = want_heldout ? bp : 10000u - bp;  // of 10000
  return keep > 1250u ? keep - 1250u : 0u;
}

__device__ __forceinline__ unsigned long long grab_estimate(unsigned long long raw,
                                                            uint32_t share) {
  return raw * share / 10000u;
}

template <bool kCopy, bool kChunked>
__global__ void __launch_bounds__(kHashThreads, kHashBlocksPerSM)
    hash_prefix_kernel(const int32_t *__restrict__ tokens, int32_t *__restrict__ copy_dst,
                       unsigned long long *tokens_read, unsigned long long *hashed,
                       const int64_t *__restrict__ offs,
                       const uint32_t *__restrict__ sdb, const uint16_t *__restrict__ stream_bp,
                       uint32_t J, uint32_t D0, const uint32_t *__restrict__ order,
                       uint32_t *__restrict__ klen, const int32_t *cum_last,
                       const unsigned *ready, unsigned ready_at, uint32_t T, uint32_t G,
                       uint64_t hash_key, uint32_t want_heldout, unsigned long long *frontier,
                       unsigned long long *prog, uint32_t j_begin, uint32_t j_count,
                       const uint16_t *__restrict__ need_num, uint32_t need_num_all,
                       const unsigned long long *__restrict__ pre_cap) {
  pdl_wait();
  constexpr uint32_t kGrab = 8;
  const int lane = threadIdx.x & 31;
  const uint32_t warp_id = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  bool ready_seen = false;
  // streams [j_begin, j_begin + j_count) of the J.  kChunked (many streams):
  // 32 looked at a time -- the lanes read their streams' state together and
  // the warp then works only on those that still need hashing (with
  // thousands of streams most are done, and one read per stream would take
  // longer than the hashing); else one after the other
  for (uint32_t c0 = 0; c0 < j_count; c0 += (kChunked ? 32 : 1)) {
    bool live = !kChunked;
    if (kChunked) {
    if (lane == 0 && !ready_seen &&
        *reinterpret_cast<const volatile unsigned *>(ready) >= ready_at) {
      __threadfence();
      ready_seen = true;
    }
    ready_seen = __shfl_sync(0xffffffffu, ready_seen, 0);
    if (c0 + lane < j_count) {
      const uint32_t j_l = j_begin + (warp_id + c0 + lane) % j_count;
      if (stream_bp[j_l] != 0) {
        const uint64_t n_l = sdb[j_l + 1] - sdb[j_l];
        const unsigned long long fr = *reinterpret_cast<volatile unsigned long long *>(frontier + j_l);
        const unsigned long long w = *reinterpret_cast<volatile unsigned long long *>(prog + j_l);
        const unsigned long long lim =
            ready_seen ? (unsigned long long)tokens_needed(
                             *reinterpret_cast<const volatile int32_t *>(cum_last + j_l), G, T,
                             need_num ? need_num[j_l] : need_num_all)
                       : (pre_cap ? pre_cap[j_l] : ~0ull);
        live = fr < n_l && (w >> 16) <= lim;
      }
    }
    }
    for (unsigned m = kChunked ? __ballot_sync(0xffffffffu, live) : 1u; m; m &= m - 1) {
    const uint32_t j = j_begin + (warp_id + c0 + (uint32_t)(__ffs(m) - 1)) % j_count;
    const uint32_t bp = stream_bp[j];
    if (!kChunked && bp == 0) continue;
    const uint64_t N = sdb[j + 1] - sdb[j];
    const uint64_t base_pos = (uint64_t)sdb[j] - D0;
    // need_j is known once the quota kernel (on another stream) has written
    // the last row of its table; until then the stream is hashed up to an
    // estimate of it from the recipe (pre_cap; none: on)
    unsigned long long need = ~0ull;
    const unsigned long long cap = pre_cap ? pre_cap[j] : ~0ull;
    while (true) {
      unsigned long long base = 0;
      if (lane == 0) {
        if (need == ~0ull) {
          if (!ready_seen && *reinterpret_cast<const volatile unsigned *>(ready) >= ready_at) {
            __threadfence();
            ready_seen = true;
          }
          if (ready_seen)
            need = (unsigned long long)tokens_needed(
                *reinterpret_cast<const volatile int32_t *>(cum_last + j), G, T,
                need_num ? need_num[j] : need_num_all);
        }
        const unsigned long long w = *reinterpret_cast<volatile unsigned long long *>(prog + j);
        const unsigned long long lim = ready_seen ? need : cap;
        base = ((w >> 16) <= lim) ? atomicAdd(frontier + j, (unsigned long long)kGrab) : N;
      }
      base = __shfl_sync(0xffffffffu, base, 0);
      if (base >= N) break;
      const uint64_t pend = min((uint64_t)N, (uint64_t)base + kGrab);
      // lanes 0..kGrab-1 fetch the grabbed positions' lengths, documents and
      // first-token offsets together, then the warp hashes them one by one
      uint32_t L_l = 0;
      int64_t o_l = 0;
      if (lane < (int)(pend - base)) {
        const uint64_t idx = base_pos + base + lane;
        L_l = klen[idx];
        if (L_l) o_l = __ldg(offs + order[idx]);
      }
      // the grab is in flight until its decisions are counted
      const uint32_t share = grab_share(bp, want_heldout);
      if (share) {
        const unsigned long long raw = warp_sum_u64(L_l);
        if (lane == 0 && raw) atomicAdd(prog + j, (grab_estimate(raw, share) << 16) + 1);
      }
      uint64_t mine = 0;  // lane q: the token-term sum of document q
      for (int q = 0; q < (int)(pend - base); q++) {
        const uint32_t L = __shfl_sync(0xffffffffu, L_l, q);
        if (L == 0) continue;
        const int64_t o0 = __shfl_sync(0xffffffffu, o_l, q);
        const uint64_t tot = warp_doc_terms<kCopy>(tokens, copy_dst, o0, L, lane);
        if (lane == q) mine = tot;
      }
      // lane q decides document q
      unsigned long long kept_here = 0;
      if (L_l) {
        const uint64_t h = splitmix64(mine ^ splitmix64(hash_key + L_l));
        const uint32_t held = (__umul64hi(h, 10000ull) < (uint64_t)bp) ? 1u : 0u;
        if (held != want_heldout)
          klen[base_pos + base + lane] = 0;
        else
          kept_here = L_l;
      }
      kept_here = warp_sum_u64(kept_here);
      const unsigned long long raw_here = warp_sum_u64(L_l);
      const unsigned docs_here = __popc(__ballot_sync(0xffffffffu, L_l != 0));
      if (lane == 0 && raw_here) {
        if (kCopy) atomicAdd(tokens_read, raw_here);
        atomicAdd(hashed, raw_here);
        atomicAdd(hashed + 1, (unsigned long long)docs_here);
        // the kept tokens in, the estimate out, one grab fewer in flight
        // (modulo 2^64: the word's count holds this grab, so nothing
        // borrows from the tokens)
        const uint32_t sh = grab_share(bp, want_heldout);
        if (sh)
          atomicAdd(prog + j, ((kept_here - grab_estimate(raw_here, sh)) << 16) - 1ull);
        else if (kept_here)
          atomicAdd(prog + j, kept_here << 16);
      }
    }
    }
  }
}

// The fraction of its bound a stream's prefix is hashed to in the second
// round, from its measured packing fill.  A block per stream: the sample is
// the longest run of the stream's first 2048 positions whose raw tokens stay
// within the first round's need (so it depends only on lengths, and every
// document in it is decided); up to 32 lanes each pack 64 of its positions
// greedily from an empty window (T-chunks, kept lengths) and count their
// closed windows and tokens.  With W windows closed, fill = tokens / (W T)
// and need_num = 1024 * min(1, fill + 0.03 + 0.4 / sqrt(min(W, windows
// needed))); 1024 (no speculation) for a stream that needs fewer than 256
// windows or whose sample closes fewer than 256.  Only the amount hashed
// depends on it: a prefix that then holds fewer windows than needed is
// caught after packing and the context is built again with the full bound.
constexpr uint32_t kFillSample = 2048;
constexpr uint32_t kFillThreads = 1024;  // threads of a block; kFillSample a multiple
constexpr uint32_t kFillRun = 64;

__device__ __forceinline__ uint32_t raw_length(const int64_t *__restrict__ offs, uint32_t d,
                                               uint64_t n_tokens) {
  const int64_t o0 = __ldg(offs + d), o1 = __ldg(offs + d + 1);
  const bool ok = o0 >= 0 && o1 > o0 && (uint64_t)o1 <= n_tokens && o1 - o0 <= 0x7FFFFFFF;
  return ok ? (uint32_t)(o1 - o0) : 0u;
}

__global__ void __launch_bounds__(kFillThreads)
    fill_need_kernel(const uint32_t *__restrict__ sdb, uint32_t D0,
                     const uint16_t *__restrict__ stream_bp, const uint32_t *__restrict__ order,
                     const uint32_t *__restrict__ klen, const int64_t *__restrict__ offs,
                     uint64_t n_tokens, const int32_t *__restrict__ cum_last, uint32_t T,
                     uint32_t G, uint32_t first_num,
                     const unsigned long long *__restrict__ pre_cap,
                     uint16_t *__restrict__ need_num) {
  pdl_wait_then_release();
  // a block per stream: the sample's raw and kept lengths are staged in
  // shared memory by all its threads at once, then one warp decides
  __shared__ uint32_t raw_s[kFillSample], kept_s[kFillSample];
  const uint32_t j = blockIdx.x;
  const int64_t wn = windows_needed(cum_last[j], G);
  if (stream_bp[j] == 0 || wn < kSpeculateMinWindows) {
    if (threadIdx.x == 0) need_num[j] = 1024;
    return;
  }
  const uint64_t b = (uint64_t)sdb[j] - D0, N = sdb[j + 1] - sdb[j];
  const uint32_t lim = (uint32_t)(N < kFillSample ? N : kFillSample);
  // every thread's documents first, then their offsets: two rounds of reads
  constexpr uint32_t kPer = kFillSample / kFillThreads;
  uint32_t d[kPer];
#pragma unroll
  for (uint32_t q = 0; q < kPer; q++) {
    const uint32_t p = threadIdx.x + q * kFillThreads;
    d[q] = p < lim ? order[b + p] : 0u;
    if (p < lim) kept_s[p] = klen[b + p];
  }
#pragma unroll
  for (uint32_t q = 0; q < kPer; q++) {
    const uint32_t p = threadIdx.x + q * kFillThreads;
    if (p < lim) raw_s[p] = raw_length(offs, d[q], n_tokens);
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  // the first round hashed each stream to its need1, or, if its warps left
  // it before the quota table was known, to more than its cap
  int64_t need1 = tokens_needed(cum_last[j], G, T, first_num);
  if (pre_cap && (int64_t)pre_cap[j] < need1) need1 = (int64_t)pre_cap[j];
  // S: positions [0, S) whose raw tokens add up to at most need1
  uint32_t S = 0;
  int64_t acc = 0;
  for (uint32_t c0 = 0; c0 < lim; c0 += 32) {
    const uint32_t p = c0 + lane;
    int64_t incl = (p < lim) ? raw_s[p] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    incl += acc;
    const unsigned ok = __ballot_sync(0xffffffffu, p < lim && incl <= need1);
    const uint32_t cnt = __popc(ok);  // the raw sums only grow: ok is a prefix
    S = c0 + cnt;
    if (cnt < 32) break;
    acc = __shfl_sync(0xffffffffu, incl, 31);
  }
  // greedy packing of runs of 64 positions of [0, S), one run per lane
  const uint32_t runs = (S / kFillRun < 32u) ? S / kFillRun : 32u;
  uint64_t w = 0, tok = 0;
  if ((uint32_t)lane < runs) {
    uint64_t used = 0;
    for (uint32_t p = lane * kFillRun; p < (lane + 1) * kFillRun; p++) {
      const uint64_t L = kept_s[p];
      if (L == 0) continue;
      const uint64_t n = L / T, t = L % T;
      if (n > 0) {
        // a full chunk closes an open window, fills one of its own, and the
        // next chunk or tail closes that one
        w += (used > 0 ? 1 : 0) + (n - 1) + (t > 0 ? 1 : 0);
        tok += used + (uint64_t)T * (n - 1) + (t > 0 ? (uint64_t)T : 0);
        used = (t > 0) ? t : T;
      } else {
        if (used + L > T) {
          w++;
          tok += used;
          used = 0;
        }
        used += L;
      }
    }
  }
  w = warp_sum_u64(w);
  tok = warp_sum_u64(tok);
  if (lane == 0) {
    uint32_t num = 1024;
    if (w >= 256) {
      const double fill = (double)tok / ((double)w * (double)T);
      const double wmin = ((int64_t)w < wn) ? (double)w : (double)wn;
      const double f = fill + 0.03 + 0.4 / sqrt(wmin);
      num = (uint32_t)min(1024.0, ceil(f * 1024.0));
    }
    need_num[j] = (uint16_t)num;
  }
}

// The reachable prefix of every stream the hash does not read (no held-out
// rate), copied from host memory the device can address into the device
// copy.  The prefix's kept tokens, in position order, are cut into chunks
// of kCopyChunk tokens, one warp per chunk, so that a long document is
// shared by many warps: the warp finds the chunk's first position by binary
// search over the kept-length scan, then copies the part of each document
// that falls in the chunk in 16-byte blocks, four in flight per lane (the
// few tokens of neighbouring documents that share a block are written with
// the values they have).  Positions whose kept length is 0 (empty, or
// malformed offsets) hold no tokens of the chunk and are never read.
constexpr int kCopyWarps = kThreads / 32;
constexpr uint32_t kCopyChunk = 16384;

__global__ void __launch_bounds__(kThreads)
    copy_prefix_kernel(SegGrid g, const uint32_t *__restrict__ sdb, uint32_t D0,
                       const uint32_t *__restrict__ cutoff, const uint16_t *__restrict__ stream_bp,
                       const uint32_t *__restrict__ order, const uint32_t *__restrict__ klen,
                       const int64_t *__restrict__ kex, const int64_t *__restrict__ offs,
                       const int32_t *__restrict__ src, int32_t *__restrict__ dst,
                       unsigned long long *tokens_read) {
  pdl_wait_then_release();
  uint32_t j, blk;
  seg_locate(g, j, blk);
  const int lane = threadIdx.x & 31;
  const uint64_t chunk = (uint64_t)blk * kCopyWarps + (threadIdx.x >> 5);
  if (stream_bp[j] != 0) return;
  const uint64_t b = (uint64_t)sdb[j] - D0, cut = cutoff[j];
  const int64_t base = kex[b], total = kex[b + cut] - base;
  const int64_t t0 = (int64_t)chunk * kCopyChunk;
  if (t0 >= total) return;
  const int64_t t1 = min(total, t0 + (int64_t)kCopyChunk);
  // the position holding kept token t0: the last p in [0, cut) with
  // kex[b + p] - base <= t0 (zero-length positions share their successor's
  // scan value and are skipped below)
  int64_t p = last_le<int64_t, int64_t>(kex, (int64_t)b, (int64_t)(b + cut), base + t0) - (int64_t)b;
  for (; p < (int64_t)cut; p++) {
    const int64_t k0 = kex[b + p] - base;
    if (k0 >= t1) break;
    const uint32_t L = klen[b + p];
    if (L == 0) continue;
    // the part of this document inside [t0, t1), as in-document offsets
    const int64_t s0 = max(t0, k0) - k0, s1 = min(t1, k0 + (int64_t)L) - k0;
    if (s1 <= s0) continue;
    const int64_t o0 = __ldg(offs + order[b + p]) + s0;
    const int64_t a0 = o0 & ~(int64_t)3;
    const uint32_t end = (uint32_t)(s1 - s0) + (uint32_t)(o0 - a0);
    const int4 *s4 = reinterpret_cast<const int4 *>(src + a0);
    int4 *d4 = reinterpret_cast<int4 *>(dst + a0);
    for (uint32_t r = 4 * (uint32_t)lane; r < end; r += 512) {
      int4 v[4];
#pragma unroll
      for (int u = 0; u < 4; u++)
        if (r + 128 * u < end) v[u] = __ldcs(s4 + ((r + 128 * u) >> 2));
#pragma unroll
      for (int u = 0; u < 4; u++)
        if (r + 128 * u < end) d4[(r + 128 * u) >> 2] = v[u];
    }
  }
  if (lane == 0) atomicAdd(tokens_read, (unsigned long long)(t1 - t0));
}

// ---------------------------------------------------------------------------
// The shuffle: position p of stream j reads document b_j + pi_j(p), pi_j a
// 4-round balanced Feistel network over 2*half bits (half = bits / 2, bits =
// max(2, ceil(log2 N_j)) rounded up to even), walked until it lands in
// [0, N_j).  Writes the document and its length (0 if empty, or if its
// offsets are malformed -- validate_offsets_kernel reports that); documents
// the stream does not keep are zeroed afterwards by hash_prefix_kernel
// (held-out ones for training, the others for validation).  For the
// validation stream (stream_bp_heldout_mode given), a stream whose source
// holds nothing out keeps nothing.
__device__ __forceinline__ uint64_t feistel(const uint64_t k[4], uint32_t half, uint64_t mask,
                                            uint64_t x) {
  uint64_t L = x >> half, R = x & mask;
#pragma unroll
  for (int r = 0; r < 4; r++) {
    const uint64_t F = splitmix64(k[r] ^ R) & mask;
    const uint64_t nl = R;
    R = L ^ F;
    L = nl;
  }
  return (L << half) | R;
}

// Half width of the balanced Feistel domain for [0, n): bits = max(2,
// ceil(log2 n)) rounded up to even.
__device__ __forceinline__ uint32_t feistel_half(uint64_t n) {
  uint32_t bits = (n <= 1) ? 0u : (uint32_t)(64 - __clzll((long long)(n - 1)));
  if (bits < 2) bits = 2;
  bits += bits & 1u;
  return bits >> 1;
}

// p in [0, n) -> its image under the keyed network, walked back into [0, n).
__device__ __forceinline__ uint64_t feistel_walk(const uint64_t k[4], uint64_t n, uint64_t p,
                                                 int *err) {
  const uint32_t half = feistel_half(n);
  const uint64_t mask = (half >= 64) ? ~0ull : ((1ull << half) - 1);
  uint64_t y = feistel(k, half, mask, p);
  for (uint32_t it = 0; y >= n; it++) {
    if (it > (1u << 20)) {
      set_error(err, kDevWalkLimit);
      return 0;
    }
    y = feistel(k, half, mask, y);
  }
  return y;
}

// Read order of windows: rank r of stream j reads window sG + sigma(r - sG)
// within its segment s = r / G of min(G, W - sG) windows, sigma keyed by
// (seed + 1, j, s); G = 0 reads windows in order (NeuronSpark-Trainer
// README, Concepts: the windows of a segment are read in random order).
__device__ __forceinline__ uint64_t window_of_rank(uint64_t seed, uint32_t j, uint32_t G,
                                                   uint64_t W, uint64_t r, int *err) {
  if (G == 0) return r;
  const uint64_t s = r / G, b = s * G;
  const uint64_t n = min((uint64_t)G, W - b);
  uint64_t k[4];
  const uint64_t ks = splitmix64(seed + 1);
#pragma unroll
  for (int q = 0; q < 4; q++)
    k[q] = splitmix64(ks ^ splitmix64(((uint64_t)j << 40) | (s << 8) | (uint64_t)q));
  return b + feistel_walk(k, n, r - b, err);
}

// Row order of an update: slot i holds row rho_k(i), rho_k keyed by
// (seed + 2, k) over [0, B).
__device__ __forceinline__ uint32_t row_of_slot(uint64_t seed, uint32_t step, uint32_t B,
                                                uint32_t i, int *err) {
  uint64_t k[4];
  const uint64_t ks = splitmix64(seed + 2);
#pragma unroll
  for (int q = 0; q < 4; q++) k[q] = splitmix64(ks ^ splitmix64(((uint64_t)step << 8) | q));
  return (uint32_t)feistel_walk(k, B, i, err);
}

// Each thread takes kOrderPerThread positions of one stream, p0 + m * 256,
// one after the other, and every pass of its walk loop is one evaluation of
// the network for every lane: a lane whose walk lands in range records that
// document and feeds its next position into the same evaluation.  A warp
// then pays for the average walk of its positions rather than the longest.
// The documents wait in a register queue (shifted at each landing, so that
// no register array is indexed at run time); once every walk has landed,
// the offsets of all of them are read together, so their latencies overlap
// instead of adding up.
constexpr uint32_t kOrderPerThread = 8;
// The scans of the kept lengths (below) work in tiles of kScanTile positions
// of the whole position range.
constexpr int kScanWarps = 8;
constexpr int kScanRounds = 8;
constexpr int kScanTile = kScanWarps * kScanRounds * 32;

// The positions p0 + m * blockDim.x (m < kOrderPerThread, below Nb) of
// stream j: their documents and kept lengths.
__device__ __forceinline__ void order_positions(const uint64_t *__restrict__ keys, uint32_t j,
                                                uint32_t b0, uint64_t N, uint64_t Nb,
                                                uint64_t p0, const int64_t *__restrict__ offs,
                                                uint64_t n_tokens, uint32_t D0,
                                                const uint16_t *__restrict__ stream_bp_heldout_mode,
                                                uint32_t *__restrict__ order,
                                                uint32_t *__restrict__ klen, int *err) {
  const uint32_t half = feistel_half(N);
  const uint64_t mask = (half >= 64) ? ~0ull : ((1ull << half) - 1);
  uint64_t k[4];
#pragma unroll
  for (int r = 0; r < 4; r++) k[r] = keys[(size_t)j * 4 + r];
  // the positions this thread takes: p0 + m * blockDim.x for m < cnt
  const uint64_t left = (Nb - p0 + blockDim.x - 1) / blockDim.x;
  const uint32_t cnt = left < kOrderPerThread ? (uint32_t)left : kOrderPerThread;
  // walks; the documents of positions m go to q[cnt - 1 - m] (each landing
  // shifts the queue by one)
  uint32_t q[kOrderPerThread];
#pragma unroll
  for (uint32_t m = 0; m < kOrderPerThread; m++) q[m] = 0;
  uint64_t x = p0;
  uint32_t m = 0, it = 0;
  while (m < cnt) {
    uint64_t y = feistel(k, half, mask, x);
    if (y >= N && ++it > (1u << 20)) {
      set_error(err, kDevWalkLimit);
      y = 0;
    }
    if (y < N) {
#pragma unroll
      for (uint32_t u = kOrderPerThread - 1; u > 0; u--) q[u] = q[u - 1];
      q[0] = b0 + (uint32_t)y;
      x = p0 + (uint64_t)(++m) * blockDim.x;
      it = 0;
    } else {
      x = y;
    }
  }
  // every document's offsets, read together
  int64_t o0[kOrderPerThread], o1[kOrderPerThread];
#pragma unroll
  for (uint32_t u = 0; u < kOrderPerThread; u++) {
    o0[u] = 0;
    o1[u] = 0;
    if (u < cnt) {
      o0[u] = __ldg(offs + q[u]);
      o1[u] = __ldg(offs + q[u] + 1);
    }
  }
  // the validation stream of a source that holds nothing out is empty
  const bool empty = stream_bp_heldout_mode && stream_bp_heldout_mode[j] == 0;
#pragma unroll
  for (uint32_t u = 0; u < kOrderPerThread; u++) {
    if (u < cnt) {
      const uint64_t pm = p0 + (uint64_t)(cnt - 1 - u) * blockDim.x;
      const bool ok = !empty && o0[u] >= 0 && o1[u] > o0[u] && (uint64_t)o1[u] <= n_tokens &&
                      o1[u] - o0[u] <= 0x7FFFFFFF;
      const uint64_t idx = (uint64_t)b0 + pm - D0;
      order[idx] = q[u];
      klen[idx] = ok ? (uint32_t)(o1[u] - o0[u]) : 0u;
    }
  }
}

__global__ void __launch_bounds__(kThreads)
    order_kernel(SegGrid g, const uint32_t *__restrict__ sdb, const uint64_t *__restrict__ keys,
                 const int64_t *__restrict__ offs, uint64_t n_tokens, uint32_t D0,
                 const uint16_t *__restrict__ stream_bp_heldout_mode,
                 const uint32_t *__restrict__ pos_lim, uint32_t *__restrict__ order,
                 uint32_t *__restrict__ klen, int *err) {
  pdl_wait_then_release();
  // the grid strides over the layout's blocks: those wholly past a stream's
  // taken positions cost an iteration, not a block
  for (uint32_t vb = blockIdx.x; vb < g.n_blocks; vb += gridDim.x) {
    uint32_t j, blk;
    seg_locate_at(g, vb, j, blk);
    const uint32_t b0 = sdb[j];
    const uint64_t N = sdb[j + 1] - b0;  // the permutation's domain
    const uint64_t Nb = pos_lim ? pos_lim[j] : N;  // the positions taken
    if (blk == 0 && Nb < N) {
      // a stream taken only in part: its lengths past the part are 0 where
      // the scans read them -- the scan tile holding the first position past
      // the part, and the tile holding the stream's last position if that
      // tile runs into the next stream (the tiles between lie wholly past
      // the part and are skipped)
      const uint64_t g0 = (uint64_t)b0 - D0, gl = g0 + Nb, ge = g0 + N;
      const uint64_t a1 = min(ge, (gl / kScanTile + 1) * kScanTile);
      const uint64_t a2 = max(gl, (ge - 1) / kScanTile * kScanTile);
      for (uint64_t q = gl + threadIdx.x; q < a1; q += blockDim.x) klen[q] = 0;
      if (ge % kScanTile != 0)
        for (uint64_t q = max(a2, a1) + threadIdx.x; q < ge; q += blockDim.x) klen[q] = 0;
    }
    const uint64_t p0 = (uint64_t)blk * blockDim.x * kOrderPerThread + threadIdx.x;
    if (p0 < Nb) order_positions(keys, j, b0, N, Nb, p0, offs, n_tokens, D0,
                                 stream_bp_heldout_mode, order, klen, err);
    __syncthreads();  // the block's stream is looked up again
  }
}

// ---------------------------------------------------------------------------
// Exclusive scans of the kept lengths and of the piece counts ceil(L / T):
// reduce per tile, scan the tile sums, rescan each tile with its offset.  A
// warp owns a contiguous run of 32 * kScanRounds elements and scans it with
// shuffles, round by round, so every load and store is coalesced.

// Tiles of the scans that lie wholly inside the unshuffled part of a stream
// shuffled only in part: positions (b_j + pos_lim_j, e_j) of stream j, whose
// lengths are 0 and whose prefix sums nothing reads (the cutoff reads them
// up to b_j + pos_lim_j, and at the stream's end, which is the next
// stream's start).  The scans neither read nor write them.
__device__ __forceinline__ bool scan_tile_skipped(const uint32_t *__restrict__ sdb, uint32_t J,
                                                  uint32_t D0,
                                                  const uint32_t *__restrict__ pos_lim,
                                                  uint64_t n, uint64_t t) {
  const uint64_t t0 = t * kScanTile, t1 = min(n, t0 + kScanTile);
  // the stream holding position t0: the last j whose range starts at or
  // before it (empty streams sharing that start come first)
  uint32_t lo = 0, hi = J;  // invariant: sdb[lo] - D0 <= t0
  while (hi - lo > 1) {
    const uint32_t mid = lo + (hi - lo) / 2;
    if ((uint64_t)(sdb[mid] - D0) <= t0)
      lo = mid;
    else
      hi = mid;
  }
  const uint64_t b = sdb[lo] - D0, e = sdb[lo + 1] - D0;
  return t0 >= b + (uint64_t)pos_lim[lo] + 1 && t1 <= e;
}

// Sums of every tile (with pos_lim, tiles wholly past a stream's shuffled
// part are marked in tile_zero and sum to 0).  With `done` (zeroed before),
// the last block to finish then turns the tile sums into their exclusive
// prefix in place and writes the totals, as scan_tiles_kernel does.
__global__ void __launch_bounds__(kScanWarps * 32)
    scan_reduce_kernel(const uint32_t *__restrict__ klen, uint64_t n, uint64_t nb, uint32_t T,
                       const uint32_t *__restrict__ sdb, uint32_t J, uint32_t D0,
                       const uint32_t *__restrict__ pos_lim, uint8_t *__restrict__ tile_zero,
                       int64_t *bs_a, int64_t *bs_b, unsigned *done, int64_t *tot_a,
                       int64_t *tot_b) {
  pdl_wait_then_release();
  __shared__ int64_t sa[kScanWarps], sb[kScanWarps];
  __shared__ bool s_skip;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the grid strides over the tiles (a tile past a stream's shuffled part
  // costs an iteration, not a block)
  for (uint64_t t = blockIdx.x; t < nb; t += gridDim.x) {
    if (pos_lim) {
      if (threadIdx.x == 0) {
        s_skip = scan_tile_skipped(sdb, J, D0, pos_lim, n, t);
        tile_zero[t] = s_skip ? 1 : 0;
      }
      __syncthreads();
      const bool skip = s_skip;
      __syncthreads();
      if (skip) {
        if (threadIdx.x == 0) {
          bs_a[t] = 0;
          bs_b[t] = 0;
        }
        continue;
      }
    }
    const uint64_t seg = t * kScanTile + (uint64_t)w * kScanRounds * 32;
    int64_t a = 0, b = 0;
#pragma unroll
    for (int r = 0; r < kScanRounds; r++) {
      const uint64_t i = seg + (uint64_t)r * 32 + lane;
      if (i < n) {
        const uint32_t v = klen[i];
        a += v;
        b += ((uint64_t)v + T - 1) / T;
      }
    }
    a = warp_sum_i64(a);
    b = warp_sum_i64(b);
    if (lane == 0) {
      sa[w] = a;
      sb[w] = b;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int64_t ta = 0, tb = 0;
      for (int q = 0; q < kScanWarps; q++) {
        ta += sa[q];
        tb += sb[q];
      }
      bs_a[t] = ta;
      bs_b[t] = tb;
    }
    __syncthreads();
  }
  if (!done || !last_block_done(done)) return;
  __shared__ int64_t ws[33];
  int64_t carry_a = 0, carry_b = 0;
  for (uint64_t c0 = 0; c0 < nb; c0 += blockDim.x) {
    const uint64_t i = c0 + threadIdx.x;
    const int64_t va = (i < nb) ? __ldcg(bs_a + i) : 0, vb = (i < nb) ? __ldcg(bs_b + i) : 0;
    int64_t ta, tb;
    const int64_t ea = block_excl_scan(va, ws, &ta);
    const int64_t eb = block_excl_scan(vb, ws, &tb);
    if (i < nb) {
      bs_a[i] = carry_a + ea;
      bs_b[i] = carry_b + eb;
    }
    carry_a += ta;
    carry_b += tb;
  }
  if (threadIdx.x == 0) {
    *tot_a = carry_a;
    *tot_b = carry_b;
  }
}

__device__ __forceinline__ int64_t warp_incl_scan(int64_t x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// One block: exclusive scan of the tile sums in place; totals to *tot_a/b.
__global__ void __launch_bounds__(1024)
    scan_tiles_kernel(int64_t *bs_a, int64_t *bs_b, uint32_t nb, int64_t *tot_a, int64_t *tot_b) {
  pdl_wait_then_release();
  __shared__ int64_t wa[32], wb[32];
  __shared__ int64_t carry_a, carry_b;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) carry_a = carry_b = 0;
  __syncthreads();
  for (uint32_t c0 = 0; c0 < nb; c0 += 1024) {
    const uint32_t i = c0 + threadIdx.x;
    const int64_t va = (i < nb) ? bs_a[i] : 0, vb = (i < nb) ? bs_b[i] : 0;
    const int64_t xa = warp_incl_scan(va, lane), xb = warp_incl_scan(vb, lane);
    if (lane == 31) {
      wa[w] = xa;
      wb[w] = xb;
    }
    __syncthreads();
    if (w == 0) {
      const int64_t ya = warp_incl_scan(wa[lane], lane), yb = warp_incl_scan(wb[lane], lane);
      wa[lane] = ya;
      wb[lane] = yb;
    }
    __syncthreads();
    const int64_t offa = carry_a + (w ? wa[w - 1] : 0) + xa - va;
    const int64_t offb = carry_b + (w ? wb[w - 1] : 0) + xb - vb;
    if (i < nb) {
      bs_a[i] = offa;
      bs_b[i] = offb;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry_a += wa[31];
      carry_b += wb[31];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *tot_a = carry_a;
    *tot_b = carry_b;
  }
}

__global__ void __launch_bounds__(kScanWarps * 32)
    scan_apply_kernel(const uint32_t *__restrict__ klen, uint64_t n, uint64_t nb, uint32_t T,
                      const uint8_t *__restrict__ tile_zero, const int64_t *__restrict__ bs_a,
                      const int64_t *__restrict__ bs_b, int64_t *__restrict__ kex,
                      int64_t *__restrict__ pex) {
  pdl_wait_then_release();
  __shared__ int64_t sa[kScanWarps], sb[kScanWarps];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the grid strides over the tiles, as in scan_reduce_kernel
  for (uint64_t t = blockIdx.x; t < nb; t += gridDim.x) {
  if (tile_zero && tile_zero[t]) continue;
  const uint64_t seg = t * kScanTile + (uint64_t)w * kScanRounds * 32;
  int64_t a = 0, b = 0;
#pragma unroll
  for (int r = 0; r < kScanRounds; r++) {
    const uint64_t i = seg + (uint64_t)r * 32 + lane;
    if (i < n) {
      const uint32_t v = klen[i];
      a += v;
      b += ((uint64_t)v + T - 1) / T;
    }
  }
  a = warp_sum_i64(a);
  b = warp_sum_i64(b);
  if (lane == 0) {
    sa[w] = a;
    sb[w] = b;
  }
  __syncthreads();
  int64_t ca = bs_a[t], cb = bs_b[t];
  for (int q = 0; q < w; q++) {
    ca += sa[q];
    cb += sb[q];
  }
#pragma unroll
  for (int r = 0; r < kScanRounds; r++) {
    const uint64_t i = seg + (uint64_t)r * 32 + lane;
    const uint32_t v = (i < n) ? klen[i] : 0u;
    const int64_t va = v, vb = (int64_t)(((uint64_t)v + T - 1) / T);
    const int64_t xa = warp_incl_scan(va, lane), xb = warp_incl_scan(vb, lane);
    if (i < n) {
      kex[i] = ca + xa - va;
      pex[i] = cb + xb - vb;
    }
    ca += __shfl_sync(0xffffffffu, xa, 31);
    cb += __shfl_sync(0xffffffffu, xb, 31);
  }
  __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Prefix of each stream that the horizon can reach: the shortest run of
// positions whose kept tokens exceed rmax_j * T (rmax_j = windows the horizon
// can read of stream j), or the whole stream.  Windows 0..rmax_j - 1 hold at most
// rmax_j * T tokens, so at least one piece follows them inside the prefix and
// their greedy packing is the same as over the whole stream.
// A warp per stream searches the sorted prefix sums 33 ways at a time (each
// lane probes one point, a ballot keeps the interval that holds the first
// position past the need), so the search takes about log_33 of the stream's
// length in dependent loads rather than log_2.
// The last block to finish then numbers every stream's first node --
// node_base[j] = the sum over j' < j of (pieces of j' + 1 terminal node) --
// and gathers what the host reads back besides: each stream's windows over
// the horizon (the quota table's last row) into rb[rb_rmax + j], the error
// word into rb[rb_err].
constexpr int kCutoffThreads = 128;
__global__ void __launch_bounds__(kCutoffThreads)
    cutoff_kernel(const uint32_t *__restrict__ sdb, uint32_t J, uint32_t D0,
                  const int64_t *__restrict__ kex, const int64_t *__restrict__ pex,
                  const int32_t *__restrict__ cum_last, uint32_t T, uint32_t G,
                  const uint16_t *__restrict__ need_num, const uint32_t *__restrict__ pos_lim,
                  uint32_t *__restrict__ cutoff, int64_t *npieces, int64_t *__restrict__ ptokens,
                  int64_t *__restrict__ node_base, uint32_t *__restrict__ rb, uint32_t rb_rmax,
                  uint32_t rb_err, const int *err, unsigned *done) {
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const uint32_t j = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (j < J) {
    const uint64_t b = sdb[j] - D0, e = sdb[j + 1] - D0;
    const uint64_t N = e - b;
    const int64_t base = kex[b];
    const int64_t need = tokens_needed(cum_last[j], G, T, need_num ? need_num[j] : 1024u);
    uint64_t c = N;
    if (kex[e] - base > need) {
      // the first m in [1, hi) whose prefix exceeds the need, else hi; a
      // stream shuffled only in part meets its need within that part (its
      // lengths are 0 past it, and the prefix sums there are not written)
      uint64_t lo = 1, hi = pos_lim ? min(N, (uint64_t)pos_lim[j]) : N;
      while (hi - lo > 32) {
        const uint64_t span = hi - lo;
        // 32 increasing points in [lo + 1, hi): span / 33 >= 1 apart
        const uint64_t m = lo + span * (uint64_t)(lane + 1) / 33;
        const unsigned hit = __ballot_sync(0xffffffffu, kex[b + m] - base > need);
        const int f = __ffs(hit) - 1;  // first probe past the need (-1: none)
        const uint64_t m_f = __shfl_sync(0xffffffffu, m, f < 0 ? 31 : f);
        const uint64_t m_p = __shfl_sync(0xffffffffu, m, f > 0 ? f - 1 : 0);
        if (f < 0) {
          lo = m_f + 1;
        } else {
          hi = m_f;
          if (f > 0) lo = m_p + 1;
        }
      }
      const uint64_t m = lo + (uint64_t)lane;
      const unsigned hit = __ballot_sync(0xffffffffu, m < hi && kex[b + m] - base > need);
      c = hit ? lo + (uint64_t)(__ffs(hit) - 1) : hi;
    }
    if (lane == 0) {
      cutoff[j] = (uint32_t)c;
      npieces[j] = pex[b + c] - pex[b];
      ptokens[j] = kex[b + c] - base;
    }
  }
  if (!last_block_done(done)) return;
  __shared__ int64_t ws[33];
  int64_t carry = 0;
  for (uint32_t c0 = 0; c0 < J; c0 += blockDim.x) {
    const uint32_t jj = c0 + threadIdx.x;
    int64_t total;
    const int64_t x = block_excl_scan((jj < J) ? __ldcg(npieces + jj) + 1 : 0, ws, &total);
    if (jj < J) {
      node_base[jj] = carry + x;
      rb[rb_rmax + jj] = (uint32_t)cum_last[jj];
    }
    carry += total;
  }
  if (threadIdx.x == 0) {
    node_base[J] = carry;
    rb[rb_err] = (uint32_t)*reinterpret_cast<const volatile int *>(err);
  }
}

// ---------------------------------------------------------------------------
// Pieces: the kept document at position p becomes ceil(L / T) pieces, T-chunks
// from its start; node k of stream j holds the source index of its first
// token, its document, its loss-mask threshold relative to the piece, and S,
// the kept tokens of the stream before it.  The stream's last node is a
// terminal with S = the prefix's kept tokens.
__global__ void __launch_bounds__(kThreads)
    expand_kernel(SegGrid g, const uint32_t *__restrict__ sdb, uint32_t D0,
                  const uint32_t *__restrict__ cutoff, const uint32_t *__restrict__ order,
                  const uint32_t *__restrict__ klen, const int64_t *__restrict__ kex,
                  const int64_t *__restrict__ pex, const int64_t *__restrict__ node_base,
                  const int64_t *__restrict__ npieces, const int64_t *__restrict__ offs,
                  const int32_t *__restrict__ loss_start, uint32_t T,
                  int64_t *__restrict__ node_src, int32_t *__restrict__ node_doc,
                  int32_t *__restrict__ node_mthr, int64_t *__restrict__ node_S) {
  pdl_wait_then_release();
  uint32_t j, blk;
  seg_locate(g, j, blk);
  const uint64_t p = (uint64_t)blk * blockDim.x + threadIdx.x;
  const uint64_t b = sdb[j] - D0;
  const uint32_t c = cutoff[j];
  if (p == 0) {
    const int64_t term = node_base[j] + npieces[j];
    node_S[term] = kex[b + c] - kex[b];
    node_src[term] = 0;
    node_doc[term] = -1;
    node_mthr[term] = 0;
  }
  if (p >= c) return;
  const uint64_t idx = b + p;
  const uint32_t L = klen[idx];
  if (L == 0) return;
  const uint32_t d = order[idx];
  const uint32_t n = (uint32_t)(((uint64_t)L + T - 1) / T);
  const int64_t node0 = node_base[j] + (pex[idx] - pex[b]);
  const int64_t sb = kex[idx] - kex[b];
  const int64_t o = offs[d];
  const int64_t ls = loss_start ? (int64_t)loss_start[d] : 0;
  for (uint32_t q = 0; q < n; q++) {
    const int64_t node = node0 + q;
    const int64_t chunk = (int64_t)q * T;
    node_src[node] = o + chunk;
    node_doc[node] = (int32_t)d;
    int64_t th = ls - chunk;
    if (th < INT32_MIN) th = INT32_MIN;
    node_mthr[node] = (int32_t)th;
    node_S[node] = sb + chunk;
  }
}

// next(q) = the last node q' in (q, terminal] with S[q'] - S[q] <= T: the
// start of the window after a window that starts at q.
__global__ void __launch_bounds__(kThreads)
    next_kernel(SegGrid g, const int64_t *__restrict__ node_base,
                const int64_t *__restrict__ npieces, const int64_t *__restrict__ node_S,
                uint32_t T, int32_t *__restrict__ next) {
  pdl_wait_then_release();
  uint32_t j, blk;
  seg_locate(g, j, blk);
  const int64_t item = (int64_t)blk * blockDim.x + threadIdx.x;
  const int64_t first = node_base[j], term = first + npieces[j];
  const int64_t q = first + item;
  if (q > term) return;
  if (q == term) {
    next[q] = (int32_t)q;
    return;
  }
  const int64_t lim = node_S[q] + (int64_t)T;
  const int64_t hi = min(term, q + (int64_t)T);
  next[q] = (int32_t)last_le<int64_t, int64_t>(node_S, q + 1, hi + 1, lim);
}

__global__ void jump_level_kernel(const int32_t *__restrict__ up, int64_t n,
                                  int32_t *__restrict__ out) {
  pdl_wait_then_release();
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= n) return;
  out[x] = __ldg(up + __ldg(up + x));
}

// Two levels from one: with up = level l, level l + 1 is up o up and level
// l + 2 is up o up o up o up, so one launch writes both from level l alone.
__global__ void jump_two_levels_kernel(const int32_t *__restrict__ up, int64_t n,
                                       int32_t *__restrict__ out1, int32_t *__restrict__ out2) {
  pdl_wait_then_release();
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= n) return;
  const int32_t b = __ldg(up + __ldg(up + x));
  out1[x] = b;
  out2[x] = __ldg(up + __ldg(up + b));
}

// W_j: hops from the stream's first node to its terminal, by binary lifting.
__global__ void count_windows_kernel(const int32_t *__restrict__ levels, int64_t n_nodes,
                                     uint32_t n_levels, const int64_t *__restrict__ node_base,
                                     const int64_t *__restrict__ npieces, uint32_t J,
                                     uint32_t *__restrict__ W) {
  pdl_wait_then_release();
  const uint32_t j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= J) return;
  if (npieces[j] == 0) {
    W[j] = 0;
    return;
  }
  const int64_t term = node_base[j] + npieces[j];
  int64_t x = node_base[j];
  uint64_t m = 0;
  for (int l = (int)n_levels - 1; l >= 0; l--) {
    const int64_t y = levels[(size_t)l * n_nodes + x];
    if (y != term) {
      x = y;
      m += 1ull << l;
    }
  }
  W[j] = (uint32_t)(m + 1);
}

// Window r of stream j starts at next^r(first): r's bits select the levels.
__global__ void __launch_bounds__(kThreads)
    window_starts_kernel(SegGrid g, const int32_t *__restrict__ levels, int64_t n_nodes,
                         uint32_t n_levels, const int64_t *__restrict__ node_base,
                         const uint32_t *__restrict__ W, const int64_t *__restrict__ wbase,
                         int32_t *__restrict__ win_start) {
  pdl_wait_then_release();
  uint32_t j, blk;
  seg_locate(g, j, blk);
  const uint64_t r = (uint64_t)blk * blockDim.x + threadIdx.x;
  if (r >= (uint64_t)(wbase[j + 1] - wbase[j])) return;
  int32_t s = -1;
  if (r < W[j]) {
    int64_t x = node_base[j];
    for (uint32_t l = 0; l < n_levels; l++)
      if ((r >> l) & 1) x = levels[(size_t)l * n_nodes + x];
    s = (int32_t)x;
  }
  win_start[wbase[j] + r] = s;
}

// The window of every row of every update of the horizon, as (first piece,
// end piece, offset of the window's first token inside its first piece).
// Rows of an update
// are ordered by stream, then by rank (or shuffled: slot i holds row
// rho_k(i)): row c belongs to the stream whose row range [rb[k][j],
// rb[k][j+1]) holds it and takes that stream's rank cum[k][j] + (c -
// rb[k][j]), which reads window window_of_rank(...); the window ends where the
// next one starts.
__device__ __forceinline__ void row_window(uint64_t x, const int32_t *__restrict__ rb,
                                           const int32_t *__restrict__ cum,
                                           const uint32_t *__restrict__ W,
                                           const int64_t *__restrict__ wbase,
                                           const int32_t *__restrict__ win_start,
                                           const int32_t *__restrict__ next,
                                           const int32_t *__restrict__ win_end,
                                           const int32_t *__restrict__ win_clip, uint32_t J,
                                           uint32_t B, uint64_t seed, uint32_t G,
                                           uint32_t shuffle_rows, int4 *__restrict__ row_win,
                                           int *err) {
  const uint32_t k = (uint32_t)(x / B), slot = (uint32_t)(x % B);
  const int32_t *rbk = rb + (size_t)k * (J + 1);
  const uint32_t Bk = (uint32_t)rbk[J];  // rows of this update (a schedule may vary them)
  int4 w = make_int4(-1, -1, 0, 0);
  if (slot < Bk) {
    const uint32_t i = shuffle_rows ? row_of_slot(seed, k, Bk, slot, err) : slot;
    const int64_t j = last_le<int32_t, int64_t>(rbk, 0, (int64_t)J, (int32_t)i);
    const int64_t r = (int64_t)cum[(size_t)k * J + j] + ((int64_t)i - rbk[j]);
    if (r < (int64_t)W[j]) {
      const uint64_t wi = window_of_rank(seed, (uint32_t)j, G, W[j], (uint64_t)r, err);
      const int64_t e = wbase[j] + (int64_t)wi;
      const int32_t st = win_start[e];
      // greedy windows end where the next one starts; wrap windows carry
      // their end and the offset of their first token inside their first piece
      w = win_end ? make_int4(st, win_end[e], win_clip[e], 0) : make_int4(st, next[st], 0, 0);
    }
  }
  row_win[x] = w;
}

// Wrap packing: the stream's kept tokens cut into windows of exactly T.  W_j
// counts the stream's windows, the last one partial, when the whole stream was
// expanded; otherwise only the windows that lie wholly inside the prefix.
__global__ void wrap_count_kernel(const int64_t *__restrict__ node_base,
                                  const int64_t *__restrict__ npieces,
                                  const int64_t *__restrict__ node_S,
                                  const uint32_t *__restrict__ cutoff,
                                  const uint32_t *__restrict__ sdb, uint32_t J, uint32_t T,
                                  uint32_t *__restrict__ W) {
  pdl_wait_then_release();
  const uint32_t j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= J) return;
  const int64_t first = node_base[j], term = first + npieces[j];
  const int64_t total = node_S[term] - node_S[first];
  const bool complete = cutoff[j] == sdb[j + 1] - sdb[j];
  W[j] = (uint32_t)(complete ? (total + T - 1) / T : total / T);
}

// Window w of a stream under wrap packing: tokens [wT, min((w+1)T, total)) of
// its kept run; its first piece is the last one starting at or before wT
// (clip = how far into it the window starts), its end the first piece
// starting at or after the window's last token + 1.
__global__ void __launch_bounds__(kThreads)
    wrap_windows_kernel(SegGrid g, const int64_t *__restrict__ node_base,
                        const int64_t *__restrict__ npieces, const int64_t *__restrict__ node_S,
                        const uint32_t *__restrict__ W, const int64_t *__restrict__ wbase,
                        uint32_t T, int32_t *__restrict__ win_start,
                        int32_t *__restrict__ win_end, int32_t *__restrict__ win_clip) {
  pdl_wait_then_release();
  uint32_t j, blk;
  seg_locate(g, j, blk);
  const uint64_t w = (uint64_t)blk * blockDim.x + threadIdx.x;
  if (w >= (uint64_t)(wbase[j + 1] - wbase[j])) return;
  const int64_t e = wbase[j] + (int64_t)w;
  if (w >= W[j]) {
    win_start[e] = win_end[e] = -1;
    win_clip[e] = 0;
    return;
  }
  const int64_t first = node_base[j], term = first + npieces[j];
  const int64_t s0 = node_S[first];
  const int64_t total = node_S[term] - s0;
  const int64_t a = (int64_t)w * T, b = min(a + (int64_t)T, total);
  const int64_t ws = last_le<int64_t, int64_t>(node_S, first, term, s0 + a);
  const int64_t we = last_le<int64_t, int64_t>(node_S, ws, term, s0 + b - 1) + 1;
  win_start[e] = (int32_t)ws;
  win_end[e] = (int32_t)we;
  win_clip[e] = (int32_t)(s0 + a - node_S[ws]);
}

// Updates [0, valid) can be assembled: up to the first bad one (the first
// that asks a stream for a window it does not have; bad_inv = K - k, 0 if
// none), or through it with drain.
__device__ __forceinline__ uint32_t valid_from(uint32_t bad_inv, uint32_t K, uint32_t drain) {
  if (bad_inv == 0) return K;
  const uint32_t f = K - bad_inv;
  return drain ? f + 1 : f;
}

// ---------------------------------------------------------------------------
// Order digest: D = splitmix64(sum_i splitmix64(x_i ^ splitmix64(i)) ^ count)
// over the item list (recipe scalars, source pairs, stream quads, the quota
// of every valid update, the first piece of every window those updates use).
__device__ __forceinline__ uint64_t digest_term(uint64_t item, uint64_t index) {
  return splitmix64(item ^ splitmix64(index));
}

__device__ __forceinline__ void digest_accumulate(uint64_t term, unsigned long long *acc) {
  __shared__ uint64_t scratch[33];
  const uint64_t s = block_sum<uint64_t>(term, scratch);
  if (threadIdx.x == 0) atomicAdd(acc, (unsigned long long)s);
}

// Term of item i of the recipe part (items [0, h0)) and of the quota of every
// valid update (items h0 + k J + j); 0 past them.
__device__ __forceinline__ uint64_t digest_item_term(const DigestHeader &h,
                                                     const int32_t *__restrict__ quota,
                                                     uint32_t K, uint32_t v, uint64_t i) {
  const uint64_t n_fixed = (uint64_t)kDigestScalars + 2ull * h.S + 4ull * h.J;
  const uint64_t h0 = n_fixed + h.n_piece_items;
  if (i < h0) {
    uint64_t x;
    if (i < kDigestScalars) {
      x = (i == 3) ? (uint64_t)v : h.scalars[i];
    } else if (i < kDigestScalars + 2ull * h.S) {
      const uint64_t q = i - kDigestScalars, s = q >> 1;
      x = (q & 1) ? (uint64_t)h.source_bp[s] : (uint64_t)h.source_weight[s];
    } else if (i >= n_fixed) {
      x = h.piece_items[i - n_fixed];
    } else {
      const uint64_t q = i - kDigestScalars - 2ull * h.S, j = q >> 2;
      switch (q & 3) {
        case 0: x = h.sdb[j]; break;
        case 1: x = h.sdb[j + 1]; break;
        case 2: x = h.ssrc[j]; break;
        default: x = h.tw[j]; break;
      }
    }
    return digest_term(x, i);
  }
  if (i - h0 < (uint64_t)K * h.J && (i - h0) / h.J < v)
    return digest_term((uint64_t)quota[i - h0], i);
  return 0;
}

// The row table in its first n_row_blocks blocks (one thread a row of an
// update); in the others, the first update that asks a stream for a window
// it does not have (one thread per (update, stream): atomicMax of K - k into
// *bad_inv, zeroed before).  The last block to finish then writes the valid
// horizon (*valid) and the first item of each stream's used windows in the
// digest, ubase[j] (a scan of min(cum[valid][j], W[j])).
__global__ void __launch_bounds__(kThreads)
    row_table_kernel(uint32_t n_row_blocks, const int32_t *__restrict__ rb,
                     const int32_t *__restrict__ cum, const uint32_t *__restrict__ W,
                     const int64_t *__restrict__ wbase, const int32_t *__restrict__ win_start,
                     const int32_t *__restrict__ next, const int32_t *__restrict__ win_end,
                     const int32_t *__restrict__ win_clip, uint32_t J, uint32_t B, uint32_t K,
                     uint64_t seed, uint32_t G, uint32_t shuffle_rows, int4 *__restrict__ row_win,
                     int *err, uint32_t *bad_inv, uint32_t drain, uint32_t *__restrict__ valid,
                     int64_t *__restrict__ ubase, unsigned *done) {
  pdl_wait_then_release();
  if (blockIdx.x < n_row_blocks) {
    const uint64_t x = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x < (uint64_t)K * B)
      row_window(x, rb, cum, W, wbase, win_start, next, win_end, win_clip, J, B, seed, G,
                 shuffle_rows, row_win, err);
  } else {
    const uint64_t i = (uint64_t)(blockIdx.x - n_row_blocks) * blockDim.x + threadIdx.x;
    if (i < (uint64_t)K * J) {
      const uint32_t k = (uint32_t)(i / J), j = (uint32_t)(i % J);
      if ((uint32_t)cum[(size_t)(k + 1) * J + j] > W[j]) atomicMax(bad_inv, K - k);
    }
  }
  if (!last_block_done(done)) return;
  __shared__ int64_t ws[33];
  const uint32_t v = valid_from(*reinterpret_cast<volatile uint32_t *>(bad_inv), K, drain);
  if (threadIdx.x == 0) *valid = v;
  int64_t carry = 0;
  for (uint32_t c0 = 0; c0 < J; c0 += blockDim.x) {
    const uint32_t j = c0 + threadIdx.x;
    int64_t u = 0;
    if (j < J) u = min((int64_t)cum[(size_t)v * J + j], (int64_t)W[j]);
    int64_t total;
    const int64_t e = block_excl_scan(u, ws, &total);
    if (j < J) ubase[j] = carry + e;
    carry += total;
  }
  if (threadIdx.x == 0) ubase[J] = carry;
}

// The order digest in one launch: its first n_item_blocks blocks sum the
// terms of the recipe and quota items, the others (a segmented grid over the
// streams' used windows) the first piece of every window the valid updates
// use; each block adds its sum into acc[0].  The last block to finish then
// writes D = splitmix64(acc ^ count) and gathers what the host reads back
// besides: each stream's window count into rb[rb_W + j], the error word into
// rb[rb_err].
__global__ void __launch_bounds__(kThreads)
    digest_kernel(uint32_t n_item_blocks, DigestHeader h, const int32_t *__restrict__ quota,
                  uint32_t K, SegGrid wg, const int64_t *__restrict__ wbase,
                  const int32_t *__restrict__ win_start, const int64_t *__restrict__ node_src,
                  const int32_t *__restrict__ node_doc, const int64_t *__restrict__ offs,
                  const uint32_t *valid, const int64_t *ubase, const uint32_t *__restrict__ W,
                  uint64_t seed, uint32_t G, const int32_t *__restrict__ win_clip, int *err,
                  unsigned long long *acc, uint64_t *digest, uint32_t *__restrict__ rb,
                  uint32_t rb_W, uint32_t rb_err, unsigned *done) {
  pdl_wait_then_release();
  const uint64_t h0 = (uint64_t)kDigestScalars + 2ull * h.S + 4ull * h.J + h.n_piece_items;
  const uint32_t J = h.J;
  const uint32_t v = *valid;
  uint64_t term = 0;
  if (blockIdx.x < n_item_blocks) {
    term = digest_item_term(h, quota, K, v, (uint64_t)blockIdx.x * blockDim.x + threadIdx.x);
  } else {
    uint32_t j, blk;
    seg_locate_at(wg, blockIdx.x - n_item_blocks, j, blk);
    const uint64_t r = (uint64_t)blk * blockDim.x + threadIdx.x;
    const uint64_t U = (uint64_t)(ubase[j + 1] - ubase[j]);
    if (r < U) {
      const uint64_t wi = window_of_rank(seed, j, G, W[j], r, err);
      const int64_t e = wbase[j] + (int64_t)wi;
      const int32_t node = win_start[e];
      const int32_t d = node_doc[node];
      const int64_t off = node_src[node] - offs[d] + (win_clip ? win_clip[e] : 0);
      const uint64_t x = ((uint64_t)(uint32_t)d << 32) | ((uint64_t)off & 0xFFFFFFFFull);
      term = digest_term(x, h0 + (uint64_t)v * J + (uint64_t)ubase[j] + r);
    }
  }
  digest_accumulate(term, acc);
  if (!last_block_done(done)) return;
  if (threadIdx.x == 0) {
    const uint64_t count = h0 + (uint64_t)v * J + (uint64_t)ubase[J];
    *digest = splitmix64((uint64_t)*reinterpret_cast<volatile unsigned long long *>(acc) ^ count);
    rb[rb_err] = (uint32_t)*reinterpret_cast<const volatile int *>(err);
  }
  for (uint32_t j = threadIdx.x; j < J; j += blockDim.x) rb[rb_W + j] = W[j];
}

}  // namespace

// ===========================================================================
// launchers
uint64_t &launch_counter() {
  static thread_local uint64_t n = 0;
  return n;
}
cudaError_t launch_validate_offsets(const int64_t *offs, uint32_t n_docs, uint64_t n_tokens,
                                    int *err, int n_sms, cudaStream_t st) {
  ++launch_counter();
  // four CTAs of eight warps per SM at most, striding over runs of 128
  const uint64_t runs = (uint64_t)n_docs / kValidateRun + 1;
  const uint64_t want = (runs + kThreads / 32 - 1) / (kThreads / 32);
  const uint32_t grid = (uint32_t)std::min<uint64_t>(want, (uint64_t)n_sms * 4);
  pdl_launch(validate_offsets_kernel, grid, kThreads, 0, st, offs, n_docs, n_tokens, err);
  return cudaGetLastError();
}

cudaError_t launch_keys_bound(uint64_t seed, uint32_t J, uint64_t *keys, const uint32_t *sdb,
                              const int64_t *offs, const uint16_t *stream_bp,
                              const unsigned long long *est_tok, uint32_t *pos_lim,
                              cudaStream_t st) {
  ++launch_counter();
  pdl_launch(keys_bound_kernel, blocks_for((uint64_t)J * 4), kThreads, 0, st, seed, J, keys, sdb,
             offs, stream_bp, est_tok, pos_lim);
  return cudaGetLastError();
}

// Threads of a block-level quota kernel over n children: whole warps, and a
// power of two once the children are ranked by sorting.
static unsigned round_warps(uint32_t n) {
  unsigned t = ((n + 31) / 32) * 32;
  if (t < 32) t = 32;
  if (n > (uint32_t)kRankDirect) {
    unsigned p = 32;
    while (p < n) p <<= 1;
    t = p;
  }
  return t;
}

cudaError_t launch_quota_sources(QuotaPieces q, uint32_t S, uint32_t K, int32_t *src_quota,
                                 cudaStream_t st) {
  ++launch_counter();
  pdl_launch(quota_sources_kernel, 1, round_warps(S), 0, st, q, S, K, src_quota);
  return cudaGetLastError();
}

cudaError_t launch_quota_strata(QuotaPieces q, const int32_t *src_quota,
                                const uint32_t *src_first, uint32_t S, uint32_t J, uint32_t K,
                                uint32_t max_strata, int32_t *quota, int32_t *cum,
                                unsigned *ready, cudaStream_t st) {
  ++launch_counter();
  pdl_launch(quota_strata_kernel, S, round_warps(max_strata), 0, st, q, src_quota, src_first, S, J, K,
                                                             quota, cum, ready);
  return cudaGetLastError();
}

template <int SMAX>
static void launch_quota_warp_s(QuotaPieces q, uint32_t S, const uint32_t *src_first, uint32_t J,
                                uint32_t K, uint32_t max_strata, int32_t *quota, int32_t *cum,
                                unsigned *ready, cudaStream_t st) {
  if (max_strata <= 1)
    pdl_launch(quota_warp_kernel<SMAX, 1>, S, 32, 0, st, q, S, src_first, J, K, quota, cum, ready);
  else if (max_strata <= 4)
    pdl_launch(quota_warp_kernel<SMAX, 4>, S, 32, 0, st, q, S, src_first, J, K, quota, cum, ready);
  else if (max_strata <= 8)
    pdl_launch(quota_warp_kernel<SMAX, 8>, S, 32, 0, st, q, S, src_first, J, K, quota, cum, ready);
  else
    pdl_launch(quota_warp_kernel<SMAX, 32>, S, 32, 0, st, q, S, src_first, J, K, quota, cum, ready);
}

cudaError_t launch_quota_warp(QuotaPieces q, uint32_t S, const uint32_t *src_first, uint32_t J,
                              uint32_t K, uint32_t max_strata, int32_t *quota, int32_t *cum,
                              unsigned *ready, cudaStream_t st) {
  ++launch_counter();
  if (S <= 4)
    launch_quota_warp_s<4>(q, S, src_first, J, K, max_strata, quota, cum, ready, st);
  else if (S <= 8)
    launch_quota_warp_s<8>(q, S, src_first, J, K, max_strata, quota, cum, ready, st);
  else if (S <= 16)
    launch_quota_warp_s<16>(q, S, src_first, J, K, max_strata, quota, cum, ready, st);
  else
    launch_quota_warp_s<32>(q, S, src_first, J, K, max_strata, quota, cum, ready, st);
  return cudaGetLastError();
}

cudaError_t launch_row_base(const int32_t *quota, uint32_t J, uint32_t K, int32_t *rb,
                            cudaStream_t st) {
  ++launch_counter();
  pdl_launch(row_base_kernel, K, (J <= 32 ? 32 : J <= 128 ? 128 : 256), 0, st, quota, J, rb);
  return cudaGetLastError();
}

cudaError_t launch_hash_prefix(const int32_t *tokens, int32_t *copy_dst,
                               unsigned long long *tokens_read, unsigned long long *hashed,
                               const int64_t *offs,
                               const uint32_t *sdb, const uint16_t *stream_bp, uint32_t J,
                               uint32_t D0, const uint32_t *order, uint32_t *klen,
                               const int32_t *cum_last, const unsigned *ready, unsigned ready_at,
                               uint32_t T, uint32_t G, uint64_t hash_key, uint32_t want_heldout,
                               unsigned long long *frontier, unsigned long long *prog,
                               uint32_t j_begin, uint32_t j_count, const uint16_t *need_num,
                               uint32_t need_num_all, const unsigned long long *pre_cap,
                               int n_sms, cudaStream_t st) {
  if (j_count == 0) return cudaSuccess;
  ++launch_counter();
  // more streams than this: the warps look at them 32 at a time
  constexpr uint32_t kChunkFrom = 64;
  // at most one grab in flight a warp: fewer warps than the progress word's
  // 16-bit count holds
  constexpr int kMaxBlocks = 0xFFFF / (kHashThreads / 32);
  const dim3 grid(min(n_sms * kHashBlocksPerSM, kMaxBlocks)), block(kHashThreads);
#define NS_HASH_LAUNCH(COPY, CHUNK)                                                          \
  pdl_launch(hash_prefix_kernel<COPY, CHUNK>, grid, block, 0, st,                                   \
      tokens, copy_dst, tokens_read, hashed, offs, sdb, stream_bp, J, D0, order, klen,          \
      cum_last, ready, ready_at, T, G, hash_key, want_heldout, frontier, prog, j_begin,         \
      j_count, need_num, need_num_all, pre_cap)
  if (copy_dst) {
    if (j_count > kChunkFrom)
      NS_HASH_LAUNCH(true, true);
    else
      NS_HASH_LAUNCH(true, false);
  } else {
    if (j_count > kChunkFrom)
      NS_HASH_LAUNCH(false, true);
    else
      NS_HASH_LAUNCH(false, false);
  }
#undef NS_HASH_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_copy_prefix(SegGrid g, const uint32_t *sdb, uint32_t D0,
                               const uint32_t *cutoff, const uint16_t *stream_bp,
                               const uint32_t *order, const uint32_t *klen, const int64_t *kex,
                               const int64_t *offs, const int32_t *src, int32_t *dst,
                               unsigned long long *tokens_read, cudaStream_t st) {
  if (g.n_blocks == 0) return cudaSuccess;
  ++launch_counter();
  pdl_launch(copy_prefix_kernel, g.n_blocks, kThreads, 0, st, g, sdb, D0, cutoff, stream_bp, order, klen,
                                                      kex, offs, src, dst, tokens_read);
  return cudaGetLastError();
}

uint32_t order_positions_per_thread() { return kOrderPerThread; }

uint32_t copy_chunk_tokens() { return kCopyChunk; }

cudaError_t launch_fill_need(const uint32_t *sdb, uint32_t J, uint32_t D0,
                             const uint16_t *stream_bp, const uint32_t *order, const uint32_t *klen,
                             const int64_t *offs, uint64_t n_tokens, const int32_t *cum_last,
                             uint32_t T, uint32_t G, uint32_t first_num,
                             const unsigned long long *pre_cap, uint16_t *need_num,
                             cudaStream_t st) {
  if (J == 0) return cudaSuccess;
  ++launch_counter();
  pdl_launch(fill_need_kernel, J, kFillThreads, 0, st, sdb, D0, stream_bp, order, klen, offs, n_tokens, cum_last,
                                      T, G, first_num, pre_cap, need_num);
  return cudaGetLastError();
}

cudaError_t launch_order(SegGrid g, const uint32_t *sdb, const uint64_t *keys,
                         const int64_t *offs, uint64_t n_tokens, uint32_t D0,
                         const uint16_t *stream_bp_heldout_mode, const uint32_t *pos_lim,
                         uint32_t *order, uint32_t *klen, int *err, int n_sms,
                         cudaStream_t st) {
  if (g.n_blocks == 0) return cudaSuccess;
  ++launch_counter();
  // eight blocks of 256 threads an SM at most, striding over the layout
  const unsigned grid = std::min<unsigned>(g.n_blocks, (unsigned)n_sms * 8u);
  pdl_launch(order_kernel, grid, kThreads, 0, st, g, sdb, keys, offs, n_tokens, D0,
                                                stream_bp_heldout_mode, pos_lim, order, klen,
                                                err);
  return cudaGetLastError();
}

constexpr uint64_t kScanFuseTiles = 256;

size_t scan_scratch_bytes(uint64_t n) {
  const uint64_t nb = (n + kScanTile - 1) / kScanTile;
  return (size_t)(nb + 1) * 2 * sizeof(int64_t) + (size_t)(nb + 15) / 16 * 16;
}

cudaError_t launch_scan_pieces(const uint32_t *klen, uint64_t n, uint32_t T, int64_t *kex,
                               int64_t *pex, void *scratch, size_t scratch_bytes,
                               const uint32_t *sdb, uint32_t J, uint32_t D0,
                               const uint32_t *pos_lim, unsigned *done, int n_sms,
                               cudaStream_t st) {
  const uint64_t nb = (n + kScanTile - 1) / kScanTile;
  // eight blocks of 256 threads an SM at most, striding over the tiles
  const unsigned grid = (unsigned)std::min<uint64_t>(nb, (uint64_t)n_sms * 8);
  if (scratch_bytes < scan_scratch_bytes(n)) return cudaErrorInvalidValue;
  int64_t *bs_a = static_cast<int64_t *>(scratch);
  int64_t *bs_b = bs_a + (nb + 1);
  uint8_t *tile_zero = pos_lim ? reinterpret_cast<uint8_t *>(bs_b + (nb + 1)) : nullptr;
  // up to kScanFuseTiles tiles the reduce's last block also scans the tile
  // sums (one launch fewer); beyond, a block of 1024 threads does
  const bool fuse = nb <= kScanFuseTiles;
  if (nb > 0) {
    ++launch_counter();
    pdl_launch(scan_reduce_kernel, grid, kScanWarps * 32, 0, st, klen, n, nb, T, sdb, J, D0,
               pos_lim, tile_zero, bs_a, bs_b, fuse ? done : nullptr, kex + n, pex + n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (!fuse || nb == 0) {
    ++launch_counter();
    pdl_launch(scan_tiles_kernel, 1, 1024, 0, st, bs_a, bs_b, (uint32_t)nb, kex + n, pex + n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || nb == 0) return e;
  }
  ++launch_counter();
  pdl_launch(scan_apply_kernel, grid, kScanWarps * 32, 0, st, klen, n, nb, T, tile_zero, bs_a,
             bs_b, kex, pex);
  return cudaGetLastError();
}

cudaError_t launch_cutoff(const uint32_t *sdb, uint32_t J, uint32_t D0, const int64_t *kex,
                          const int64_t *pex, const int32_t *cum_last, uint32_t T, uint32_t G,
                          const uint16_t *need_num, const uint32_t *pos_lim, uint32_t *cutoff,
                          int64_t *npieces, int64_t *ptokens, int64_t *node_base, uint32_t *rb,
                          uint32_t rb_rmax, uint32_t rb_err, const int *err, unsigned *done,
                          cudaStream_t st) {
  ++launch_counter();
  pdl_launch(cutoff_kernel, blocks_for((uint64_t)J * 32, kCutoffThreads), kCutoffThreads, 0, st, sdb, J, D0, kex,
             pex, cum_last, T, G, need_num, pos_lim, cutoff, npieces, ptokens, node_base, rb,
             rb_rmax, rb_err, err, done);
  return cudaGetLastError();
}

cudaError_t launch_expand(SegGrid g, const uint32_t *sdb, uint32_t D0, const uint32_t *cutoff,
                          const uint32_t *order, const uint32_t *klen, const int64_t *kex,
                          const int64_t *pex, const int64_t *node_base, const int64_t *npieces,
                          const int64_t *offs, const int32_t *loss_start, uint32_t T,
                          int64_t *node_src, int32_t *node_doc, int32_t *node_mthr,
                          int64_t *node_S, cudaStream_t st) {
  if (g.n_blocks == 0) return cudaSuccess;
  ++launch_counter();
  pdl_launch(expand_kernel, g.n_blocks, kThreads, 0, st, g, sdb, D0, cutoff, order, klen, kex, pex,
                                                 node_base, npieces, offs, loss_start, T,
                                                 node_src, node_doc, node_mthr, node_S);
  return cudaGetLastError();
}

cudaError_t launch_next(SegGrid g, const int64_t *node_base, const int64_t *npieces,
                        const int64_t *node_S, uint32_t T, int32_t *next, cudaStream_t st) {
  if (g.n_blocks == 0) return cudaSuccess;
  ++launch_counter();
  pdl_launch(next_kernel, g.n_blocks, kThreads, 0, st, g, node_base, npieces, node_S, T, next);
  return cudaGetLastError();
}

cudaError_t launch_jump_level(const int32_t *up_prev, int64_t n_nodes, int32_t *up_next,
                              cudaStream_t st) {
  ++launch_counter();
  pdl_launch(jump_level_kernel, blocks_for((uint64_t)n_nodes), kThreads, 0, st, up_prev, n_nodes,
                                                                         up_next);
  return cudaGetLastError();
}

cudaError_t launch_jump_two_levels(const int32_t *up_prev, int64_t n_nodes, int32_t *up_next,
                                   int32_t *up_next2, cudaStream_t st) {
  ++launch_counter();
  pdl_launch(jump_two_levels_kernel, blocks_for((uint64_t)n_nodes), kThreads, 0, st, up_prev, n_nodes,
                                                                              up_next, up_next2);
  return cudaGetLastError();
}

cudaError_t launch_count_windows(const int32_t *levels, int64_t n_nodes, uint32_t n_levels,
                                 const int64_t *node_base, const int64_t *npieces, uint32_t J,
                                 uint32_t *W, cudaStream_t st) {
  ++launch_counter();
  pdl_launch(count_windows_kernel, blocks_for(J, 128), 128, 0, st, levels, n_nodes, n_levels, node_base,
                                                           npieces, J, W);
  return cudaGetLastError();
}

cudaError_t launch_window_starts(SegGrid g, const int32_t *levels, int64_t n_nodes,
                                 uint32_t n_levels, const int64_t *node_base, const uint32_t *W,
                                 const int64_t *wbase, int32_t *win_start, cudaStream_t st) {
  if (g.n_blocks == 0) return cudaSuccess;
  ++launch_counter();
  pdl_launch(window_starts_kernel, g.n_blocks, kThreads, 0, st, g, levels, n_nodes, n_levels, node_base,
                                                        W, wbase, win_start);
  return cudaGetLastError();
}

cudaError_t launch_wrap_windows(SegGrid g, const int64_t *node_base, const int64_t *npieces,
                                const int64_t *node_S, const uint32_t *cutoff,
                                const uint32_t *sdb, uint32_t J, uint32_t T, uint32_t *W,
                                const int64_t *wbase, int32_t *win_start, int32_t *win_end,
                                int32_t *win_clip, cudaStream_t st) {
  ++launch_counter();
  pdl_launch(wrap_count_kernel, blocks_for(J, 128), 128, 0, st, node_base, npieces, node_S, cutoff, sdb,
                                                        J, T, W);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || g.n_blocks == 0) return e;
  ++launch_counter();
  pdl_launch(wrap_windows_kernel, g.n_blocks, kThreads, 0, st, g, node_base, npieces, node_S, W, wbase,
                                                       T, win_start, win_end, win_clip);
  return cudaGetLastError();
}

cudaError_t launch_row_table(const int32_t *rb, const int32_t *cum, const uint32_t *W,
                             const int64_t *wbase, const int32_t *win_start, const int32_t *next,
                             const int32_t *win_end, const int32_t *win_clip, uint32_t J,
                             uint32_t B, uint32_t K, uint64_t seed, uint32_t G,
                             uint32_t shuffle_rows, int4 *row_win, int *err, uint32_t *bad_inv,
                             uint32_t drain, uint32_t *valid, int64_t *ubase, unsigned *done,
                             cudaStream_t st) {
  ++launch_counter();
  const uint32_t n_row = blocks_for((uint64_t)K * B), n_bad = blocks_for((uint64_t)K * J);
  pdl_launch(row_table_kernel, n_row + n_bad, kThreads, 0, st, n_row, rb, cum, W, wbase,
             win_start, next, win_end, win_clip, J, B, K, seed, G, shuffle_rows, row_win, err,
             bad_inv, drain, valid, ubase, done);
  return cudaGetLastError();
}

cudaError_t launch_digest(const DigestHeader &h, const int32_t *quota, uint32_t K, SegGrid wg,
                          const int64_t *wbase, const int32_t *win_start,
                          const int64_t *node_src, const int32_t *node_doc, const int64_t *offs,
                          const uint32_t *valid, const int64_t *ubase, const uint32_t *W,
                          uint64_t seed, uint32_t G, const int32_t *win_clip, int *err,
                          unsigned long long *acc, uint64_t *digest, uint32_t *rb, uint32_t rb_W,
                          uint32_t rb_err, unsigned *done, cudaStream_t st) {
  const uint64_t h0 = (uint64_t)kDigestScalars + 2ull * h.S + 4ull * h.J + h.n_piece_items;
  const uint32_t n_items = blocks_for(h0 + (uint64_t)K * h.J);
  ++launch_counter();
  pdl_launch(digest_kernel, n_items + wg.n_blocks, kThreads, 0, st, n_items, h, quota, K, wg,
             wbase, win_start, node_src, node_doc, offs, valid, ubase, W, seed, G, win_clip, err,
             acc, digest, rb, rb_W, rb_err, done);
  return cudaGetLastError();
}

}  // namespace nsk
