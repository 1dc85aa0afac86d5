// Per-update assembly: one CTA per (update, row).  The row's window comes
// from the row table built at init; the window's pieces are staged in shared
// memory and copied in order into T positions of tokens / position ids /
// document ids / loss mask, the rest padded; the row's fingerprint and
// learned-position count are reduced in the same pass.
//
// Rows of exactly T positions, padded (Linnet training docs, Supervised
// fine-tuning); a position id of 0 starts each sequence within a row (Other
// trainers); only completion tokens are learned (Supervised fine-tuning);
// rows are a pure function of (recipe, seed, update, row), so any split of
// the rows gives the same bytes ("Zephon: deterministic data loading",
// checkpoint on 16 GPUs, resume on 8/32/64).
//
// Layout of the work: 8 warps per CTA; a warp owns tiles of 128 consecutive
// positions (4 per lane, so every store is a 16-byte vector and a warp
// writes 512 contiguous bytes per array) and handles two tiles per round,
// issuing both tiles' token loads before computing either.  A tile inside one
// piece reads its tokens with one aligned 16-byte load per lane, realigned
// across lanes with shuffles; a tile that crosses piece ends reads them one by
// one.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace nsk {

namespace {

constexpr int kGatherWarps = 8;
constexpr int kTile = 128;       // positions per warp per tile: 32 lanes x 4
constexpr int kPieceCap = 512;   // pieces of a window staged in shared memory

// Fingerprint terms of position t: key_t = a_t ^ ((b_t | t << 40) * golden),
// a_t = (u32 tok << 32) | u32 doc, b_t = (mask << 32) | u32 pos.
__device__ __forceinline__ uint64_t fp_term(int32_t tok, int32_t pos, int32_t doc, uint32_t m,
                                            uint32_t t) {
  const uint64_t a = ((uint64_t)(uint32_t)tok << 32) | (uint64_t)(uint32_t)doc;
  const uint64_t b = ((uint64_t)m << 32) | (uint64_t)(uint32_t)pos;
  return splitmix64(a ^ ((b | ((uint64_t)t << 40)) * kGolden));
}

__device__ __forceinline__ int4 shfl_down4(const int4 &v) {
  int4 r;
  r.x = __shfl_down_sync(0xffffffffu, v.x, 1);
  r.y = __shfl_down_sync(0xffffffffu, v.y, 1);
  r.z = __shfl_down_sync(0xffffffffu, v.z, 1);
  r.w = __shfl_down_sync(0xffffffffu, v.w, 1);
  return r;
}

// The window's pieces, either staged in shared memory or read from the
// context's tables.  dst(q) is the first row position of piece q (relative to
// the window), dst(np) the window's used length.
struct Pieces {
  const int64_t *S;     // staged: S - S[ws] prefix; global: node_S + ws (absolute)
  const int64_t *src;   // first token index of each piece
  const int32_t *doc;
  const int32_t *mthr;
  int64_t sbase;        // subtracted from S to make it window-relative
  int32_t np;
  __device__ __forceinline__ int64_t dst(int32_t q) const { return S[q] - sbase; }
  // last piece q in [lo, np) with dst(q) <= t (dst(lo) <= t); pieces of one
  // warp's tiles only move forward, so a few linear probes usually suffice
  __device__ __forceinline__ int32_t find(int32_t lo, int64_t t) const {
#pragma unroll
    for (int probe = 0; probe < 3; probe++) {
      if (lo + 1 >= np || S[lo + 1] - sbase > t) return lo;
      lo++;
    }
    int32_t l = lo, h = np;
    while (l < h) {
      const int32_t m = l + (h - l) / 2;
      if (S[m] - sbase <= t)
        l = m + 1;
      else
        h = m;
    }
    return l - 1;
  }
};

// cp.async: 16 bytes global -> shared, asynchronous, tracked in groups.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

constexpr int kStages = 4;         // tiles in flight per warp
constexpr int kStageWords = 132;   // 128 tokens + up to 3 of misalignment, 16-byte multiple

// What a tile needs between its copy and its stores (kept in shared memory).
struct TileMeta {
  int32_t kind;  // 0 pad, 1 inside piece q (staged), 2 crosses piece ends
  int32_t q;     // piece of the tile's first position
  int32_t x0;    // offset of the tile's first position inside piece q
  int32_t sh;    // source misalignment in tokens (kind 1)
};

// Classify tile t0 and, for a tile inside one piece, start copying its tokens
// (rounded out to 16-byte blocks that each hold at least one of them).
__device__ __forceinline__ void tile_issue(const GatherParams &p, const Pieces &P, int32_t used,
                                           uint32_t t0, int32_t q_hint, int lane, int32_t *buf,
                                           TileMeta *meta) {
  TileMeta m;
  m.kind = 0;
  m.q = q_hint;
  m.x0 = 0;
  m.sh = 0;
  if ((int32_t)t0 < used) {
    m.q = P.find(q_hint, (int64_t)t0);
    const int64_t qs = P.dst(m.q);
    const int64_t qe = P.dst(m.q + 1);
    m.x0 = (int32_t)((int64_t)t0 - qs);
    if (qe >= (int64_t)t0 + kTile) {
      m.kind = 1;
      const int64_t srcw = P.src[m.q] + m.x0;
      m.sh = (int32_t)(srcw & 3);
      const int32_t *g = p.tokens + (srcw - m.sh);
      cp_async16(buf + 4 * lane, g + 4 * lane);
      if (lane == 0 && m.sh != 0) cp_async16(buf + 128, g + 128);
    } else {
      m.kind = 2;
    }
  }
  if (lane == 0) *meta = m;
}

__device__ __forceinline__ void tile_store(const GatherParams &p, const Pieces &P, int32_t used,
                                           uint32_t t0, int lane, size_t obase, const int32_t *buf,
                                           const TileMeta &m, uint64_t &acc, int &learned) {
  const uint32_t tp = t0 + 4u * lane;
  int4 tk, ps, dc;
  uint32_t mk = 0;
  if (m.kind == 0) {
    tk = make_int4(p.pad_id, p.pad_id, p.pad_id, p.pad_id);
    ps = make_int4(0, 0, 0, 0);
    dc = make_int4(-1, -1, -1, -1);
  } else if (m.kind == 1) {
    const int4 v = *reinterpret_cast<const int4 *>(buf + 4 * lane);
    if (m.sh == 0) {
      tk = v;
    } else {
      int4 nv = shfl_down4(v);
      if (lane == 31) nv = *reinterpret_cast<const int4 *>(buf + 128);
      if (m.sh == 1)
        tk = make_int4(v.y, v.z, v.w, nv.x);
      else if (m.sh == 2)
        tk = make_int4(v.z, v.w, nv.x, nv.y);
      else
        tk = make_int4(v.w, nv.x, nv.y, nv.z);
    }
    const int32_t x = m.x0 + 4 * lane;
    ps = make_int4(x, x + 1, x + 2, x + 3);
    const int32_t d = P.doc[m.q];
    dc = make_int4(d, d, d, d);
    const int32_t th = P.mthr[m.q];
    mk = (x >= th ? 1u : 0u) | (x + 1 >= th ? 1u << 8 : 0u) | (x + 2 >= th ? 1u << 16 : 0u) |
         (x + 3 >= th ? 1u << 24 : 0u);
  } else {
    if (tp >= p.T) return;
    int32_t e0[4], e1[4], e2[4];
    int32_t qq = -1;
    int64_t qqe = 0, qqs = 0;
#pragma unroll
    for (int e = 0; e < 4; e++) {
      const int32_t t = (int32_t)tp + e;
      if (t >= used) {
        e0[e] = p.pad_id;
        e1[e] = 0;
        e2[e] = -1;
        continue;
      }
      if (qq < 0) {
        qq = P.find(m.q, (int64_t)t);
        qqs = P.dst(qq);
        qqe = P.dst(qq + 1);
      }
      while ((int64_t)t >= qqe) {
        qq++;
        qqs = qqe;
        qqe = P.dst(qq + 1);
      }
      const int32_t x = t - (int32_t)qqs;
      e0[e] = __ldg(p.tokens + P.src[qq] + x);
      e1[e] = x;
      e2[e] = P.doc[qq];
      if (x >= P.mthr[qq]) mk |= 1u << (8 * e);
    }
    tk = make_int4(e0[0], e0[1], e0[2], e0[3]);
    ps = make_int4(e1[0], e1[1], e1[2], e1[3]);
    dc = make_int4(e2[0], e2[1], e2[2], e2[3]);
  }
  if (tp >= p.T) return;
  __stcs(reinterpret_cast<int4 *>(p.tokens_out + obase + tp), tk);
  __stcs(reinterpret_cast<int4 *>(p.pos_out + obase + tp), ps);
  __stcs(reinterpret_cast<int4 *>(p.doc_out + obase + tp), dc);
  __stcs(reinterpret_cast<unsigned int *>(p.mask_out + obase + tp), mk);
  acc += fp_term(tk.x, ps.x, dc.x, mk & 1u, tp);
  acc += fp_term(tk.y, ps.y, dc.y, (mk >> 8) & 1u, tp + 1);
  acc += fp_term(tk.z, ps.z, dc.z, (mk >> 16) & 1u, tp + 2);
  acc += fp_term(tk.w, ps.w, dc.w, (mk >> 24) & 1u, tp + 3);
  learned += __popc(mk);
}

__global__ void __launch_bounds__(kGatherWarps * 32)
    gather_kernel(const GatherParams p) {
  __shared__ int64_t s_S[kPieceCap + 1];
  __shared__ int64_t s_src[kPieceCap];
  __shared__ int32_t s_doc[kPieceCap];
  __shared__ int32_t s_mthr[kPieceCap];
  __shared__ __align__(16) int32_t s_tok[kGatherWarps][kStages][kStageWords];
  __shared__ TileMeta s_meta[kGatherWarps][kStages];
  __shared__ uint64_t s_fp[kGatherWarps];
  __shared__ int s_learned[kGatherWarps];

  const uint32_t blk = blockIdx.x;
  const uint32_t step_local = blk / p.n_rows;
  const uint32_t row_local = blk - step_local * p.n_rows;
  const uint32_t k = p.step0 + step_local;
  const uint32_t i = p.row0 + row_local;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // the row's window: pieces [ws, we) of the context's piece table
  const int2 win = p.row_win[(size_t)k * p.B + i];
  int64_t ws = win.x, we = win.y;
  if (ws < 0 || we < ws) ws = we = 0;  // a row past the end of its stream: all padding
  const int32_t np = (int32_t)(we - ws);
  Pieces P;
  P.np = np;
  const bool staged = np <= kPieceCap;
  if (staged) {
    for (int32_t t = threadIdx.x; t <= np; t += blockDim.x) {
      s_S[t] = __ldg(p.node_S + ws + t);
      if (t < np) {
        s_src[t] = __ldg(p.node_src + ws + t);
        s_doc[t] = __ldg(p.node_doc + ws + t);
        s_mthr[t] = __ldg(p.node_mthr + ws + t);
      }
    }
    __syncthreads();
    P.S = s_S;
    P.src = s_src;
    P.doc = s_doc;
    P.mthr = s_mthr;
  } else {
    P.S = p.node_S + ws;
    P.src = p.node_src + ws;
    P.doc = p.node_doc + ws;
    P.mthr = p.node_mthr + ws;
  }
  P.sbase = P.S[0];
  const int64_t used64 = P.S[np] - P.sbase;
  int32_t used = (int32_t)used64;
  if (used64 < 0 || used64 > (int64_t)p.T) {
    set_error(p.err, kDevBadNode);
    used = 0;
  }

  // this warp's tiles: t0 = warp * 128 + m * 1024, m < n_tiles, through a
  // ring of kStages shared-memory buffers filled by cp.async
  constexpr uint32_t kStride = kGatherWarps * kTile;
  const uint32_t first = (uint32_t)warp * kTile;
  const int n_tiles = first < p.T ? (int)((p.T - first + kStride - 1) / kStride) : 0;
  int32_t(*ring)[kStageWords] = s_tok[warp];
  TileMeta *meta = s_meta[warp];
  int32_t q_hint = 0;
#pragma unroll
  for (int m = 0; m < kStages - 1; m++) {
    if (m < n_tiles) {
      tile_issue(p, P, used, first + m * kStride, q_hint, lane, ring[m], &meta[m]);
      __syncwarp();
      q_hint = meta[m].q;
    }
    cp_async_commit();
  }
  const size_t obase = (size_t)blk * p.T;
  uint64_t acc = 0;
  int learned = 0;
  for (int m = 0; m < n_tiles; m++) {
    const int mi = m + kStages - 1;
    if (mi < n_tiles) {
      tile_issue(p, P, used, first + mi * kStride, q_hint, lane, ring[mi % kStages],
                 &meta[mi % kStages]);
    }
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncwarp();
    if (mi < n_tiles) q_hint = meta[mi % kStages].q;
    const TileMeta mt = meta[m % kStages];
    tile_store(p, P, used, first + m * kStride, lane, obase, ring[m % kStages], mt, acc, learned);
    __syncwarp();
  }

  acc = warp_sum_u64(acc);
  learned = warp_sum_i32(learned);
  if (lane == 0) {
    s_fp[warp] = acc;
    s_learned[warp] = learned;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t a = 0;
    int l = 0;
#pragma unroll
    for (int w = 0; w < kGatherWarps; w++) {
      a += s_fp[w];
      l += s_learned[w];
    }
    p.row_fp[blk] = splitmix64(a);
    p.row_learned[blk] = l;
  }
}

// Batch fingerprint of each update: F = splitmix64(F ^ fp_i) over its rows,
// in row order.  One block per update stages the row values in shared memory
// so the serial fold never waits on global memory.
constexpr int kFoldChunk = 2048;

__global__ void __launch_bounds__(256)
    batch_fp_kernel(const uint64_t *__restrict__ row_fp, uint32_t n_rows,
                    uint64_t *__restrict__ out) {
  __shared__ uint64_t s[kFoldChunk];
  const uint64_t *f = row_fp + (size_t)blockIdx.x * n_rows;
  uint64_t F = 0;
  for (uint32_t c0 = 0; c0 < n_rows; c0 += kFoldChunk) {
    const uint32_t n = min((uint32_t)kFoldChunk, n_rows - c0);
    for (uint32_t t = threadIdx.x; t < n; t += blockDim.x) s[t] = __ldg(f + c0 + t);
    __syncthreads();
    if (threadIdx.x == 0)
      for (uint32_t t = 0; t < n; t++) F = splitmix64(F ^ s[t]);
    __syncthreads();
  }
  if (threadIdx.x == 0) out[blockIdx.x] = F;
}

}  // namespace

cudaError_t launch_gather(const GatherParams &p, cudaStream_t st) {
  const uint64_t n = (uint64_t)p.n_steps * p.n_rows;
  if (n == 0) return cudaSuccess;
  ++launch_counter();
  gather_kernel<<<(unsigned)n, kGatherWarps * 32, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_batch_fp(const uint64_t *row_fp, uint32_t n_steps, uint32_t n_rows,
                            uint64_t *out, cudaStream_t st) {
  ++launch_counter();
  batch_fp_kernel<<<n_steps, 256, 0, st>>>(row_fp, n_rows, out);
  return cudaGetLastError();
}

}  // namespace nsk
