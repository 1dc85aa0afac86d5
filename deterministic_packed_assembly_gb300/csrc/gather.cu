// Per-update assembly: one CTA per (update, row).  The row's window comes
// from the row table built at init; its pieces are copied in order into T
// positions of tokens / position ids / document ids / loss mask, the rest
// padded; the row's fingerprint and learned-position count are reduced in the
// same pass.
//
// Rows of exactly T positions, padded (Linnet training docs, Supervised
// fine-tuning); a position id of 0 starts each sequence within a row (Other
// trainers); only completion tokens are learned (Supervised fine-tuning);
// rows are a pure function of (recipe, seed, update, row), so any split of
// the rows gives the same bytes ("Zephon: deterministic data loading",
// checkpoint on 16 GPUs, resume on 8/32/64).
//
// Layout of the work: 4 warps per CTA (10 CTAs per SM; more warps and fewer
// CTAs for rows longer than 8192 positions), each on its own; a
// warp owns tiles of 128 consecutive positions (4 per lane, so every store is
// a 16-byte vector and a warp writes 512 contiguous bytes per array).  A window of up to 32
// pieces is held in the warp's registers, piece l in lane l, and looked up
// with a ballot; longer windows are read from the piece table.  Tokens of a
// tile inside one piece are copied by cp.async into a four-tile ring in
// shared memory (aligned 16-byte blocks, realigned across lanes with
// shuffles); a tile that crosses piece ends is staged token by token (4-byte
// copies into the same ring), each lane looking its positions' pieces up.
// Warps combine the row's fingerprint through shared-memory atomics and the
// last one to finish writes it, so no warp waits for another.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace nsk {

namespace {

constexpr int kTile = 128;         // positions per warp per tile: 32 lanes x 4
constexpr int kStages = 4;         // tiles in flight per warp
constexpr int kHalfStage = 132;    // 128 tokens + up to 3 of misalignment, 16-byte multiple
// Words of a ring slot: room for two runs (a tile over two pieces) with up to
// 8 warps a CTA; with 16 (rows beyond 16384 positions, whose pieces are
// long) one run, so that the CTA's shared memory stays within 48 KB, and
// such tiles are staged token by token.
template <int W>
__host__ __device__ constexpr int stage_words() {
  return W <= 8 ? 2 * kHalfStage : kHalfStage;
}

// Fingerprint term of position t: key_t = a_t ^ ((b_t | t << 40) * golden),
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

// cp.async: 16 bytes global -> shared, asynchronous, tracked in groups.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// A piece of the window: its first row position (relative to the window), the
// token index of its first token, its document and loss threshold.
struct Piece {
  int32_t start, end;
  int64_t src;
  int32_t doc, mthr;
};

// Window of at most 32 pieces held in the warp's registers: lane l holds
// piece l.  Every method is called by all 32 lanes together.
struct WarpPieces {
  int32_t S;     // start of this lane's piece, INT_MAX past the last piece
  int64_t src;
  int32_t doc, mthr;
  int32_t np, used;
  // last piece whose start is <= t, for a t the whole warp shares
  __device__ __forceinline__ int32_t find_uniform(int32_t t) const {
    return __popc(__ballot_sync(0xffffffffu, S <= t)) - 1;
  }
  // last piece whose start is <= t, for a t of this lane's own
  __device__ __forceinline__ int32_t find_lane(int32_t t) const {
    int32_t pos = 0;
#pragma unroll
    for (int step = 16; step > 0; step >>= 1) {
      const int32_t v = __shfl_sync(0xffffffffu, S, min(pos + step, 31));
      if (pos + step < 32 && v <= t) pos += step;
    }
    return pos;
  }
  __device__ __forceinline__ Piece get(int32_t q) const {
    Piece p;
    p.start = __shfl_sync(0xffffffffu, S, q);
    const int32_t nxt = __shfl_sync(0xffffffffu, S, min(q + 1, 31));
    p.end = (q + 1 < np) ? nxt : used;
    p.src = __shfl_sync(0xffffffffu, src, q);
    p.doc = __shfl_sync(0xffffffffu, doc, q);
    p.mthr = __shfl_sync(0xffffffffu, mthr, q);
    return p;
  }
};

// Loss threshold of a piece whose first `clip` tokens lie in an earlier window.
__device__ __forceinline__ int32_t clip_threshold(int32_t mthr, int32_t clip) {
  return (int32_t)max((int64_t)mthr - clip, (int64_t)INT_MIN);
}

// Window of any length read from the context's piece table (L1-cached).
struct TablePieces {
  const int64_t *S;  // node_S + ws (absolute prefix; sbase subtracted)
  const int64_t *srcs;
  const int32_t *docs, *mthrs;
  int64_t sbase;  // node_S[ws] + clip: position 0 of the row
  int32_t np, used, clip;
  __device__ __forceinline__ int32_t find(int32_t lo, int32_t t) const {
    int32_t l = lo, h = np;
    while (l < h) {
      const int32_t m = l + (h - l) / 2;
      if (__ldg(S + m) - sbase <= t)
        l = m + 1;
      else
        h = m;
    }
    return l - 1;
  }
  __device__ __forceinline__ int32_t find_uniform(int32_t t) const { return find(0, t); }
  __device__ __forceinline__ int32_t find_lane(int32_t t) const { return find(0, t); }
  __device__ __forceinline__ Piece get(int32_t q) const {
    Piece p;
    p.start = q == 0 ? 0 : (int32_t)(__ldg(S + q) - sbase);
    p.end = q + 1 < np ? (int32_t)(__ldg(S + q + 1) - sbase) : used;
    p.src = __ldg(srcs + q) + (q == 0 ? clip : 0);
    p.doc = __ldg(docs + q);
    p.mthr = q == 0 ? clip_threshold(__ldg(mthrs + q), clip) : __ldg(mthrs + q);
    return p;
  }
};

// What a tile needs between its copy and its stores.
struct TileMeta {
  int32_t kind;  // 0 pad; 1 inside one piece; 2 three or more pieces (staged token
                 // by token); 3 at most two pieces, then padding (a run of each copied)
  int32_t x0;    // offset of the tile's first position inside its (first) piece
  int32_t sh;    // source misalignment in tokens of the (first) piece's run
  int32_t doc, mthr;
  int32_t bnd;    // kind 3: tile offset where the second piece starts
  int32_t nreal;  // kind 3: real positions of the tile, the padding after them
  int32_t sh2, doc2, mthr2;  // kind 3: the second piece's run
};

// Classify tile t0 and start copying its tokens: a tile inside one piece, or
// over at most two pieces and padding, copies each piece's run rounded out
// to 16-byte blocks that each hold at least one of its tokens (the second
// run into the second half of the slot); a tile over more pieces stages its
// tokens one by one.
template <bool kTwoRuns, class PV>
__device__ __forceinline__ TileMeta tile_issue(const GatherParams &p, const PV &P, uint32_t t0,
                                               int lane, int32_t *buf) {
  TileMeta m{0, 0, 0, -1, 0, 0, 0, 0, -1, 0};
  if ((int32_t)t0 < P.used) {
    const int32_t qa = P.find_uniform((int32_t)t0);
    const Piece pc = P.get(qa);
    if (pc.end >= (int32_t)t0 + kTile) {
      m.kind = 1;
      m.x0 = (int32_t)t0 - pc.start;
      m.doc = pc.doc;
      m.mthr = pc.mthr;
      const int64_t srcw = pc.src + m.x0;
      m.sh = (int32_t)(srcw & 3);
      const int32_t *g = p.tokens + (srcw - m.sh);
      cp_async16(buf + 4 * lane, g + 4 * lane);
      if (lane == 0 && m.sh != 0) cp_async16(buf + 128, g + 128);
      return m;
    }
    // the tile's real positions end at lim; piece a holds [t0, min(end, lim))
    const int32_t lim = min((int32_t)t0 + kTile, P.used);
    const int32_t la = min(pc.end, lim) - (int32_t)t0;
    int32_t lb = 0;
    Piece pb{0, 0, 0, -1, 0};
    bool two = kTwoRuns;
    if (kTwoRuns && pc.end < lim) {
      pb = P.get(qa + 1);
      two = pb.end >= lim;
      lb = lim - pc.end;
    }
    if (two) {
      m.kind = 3;
      m.x0 = (int32_t)t0 - pc.start;
      m.doc = pc.doc;
      m.mthr = pc.mthr;
      m.bnd = la;
      m.nreal = la + lb;
      const int64_t sa = pc.src + m.x0;
      m.sh = (int32_t)(sa & 3);
      const int32_t *ga = p.tokens + (sa - m.sh);
      const int32_t na = (m.sh + la + 3) >> 2;  // at most 33 blocks
      if (lane < na) cp_async16(buf + 4 * lane, ga + 4 * lane);
      if (lane == 0 && na > 32) cp_async16(buf + 128, ga + 128);
      if (lb > 0) {
        // the second piece's run starts at its first token
        m.sh2 = (int32_t)(pb.src & 3);
        m.doc2 = pb.doc;
        m.mthr2 = pb.mthr;
        const int32_t *gb = p.tokens + (pb.src - m.sh2);
        const int32_t nb = (m.sh2 + lb + 3) >> 2;
        if (lane < nb) cp_async16(buf + kHalfStage + 4 * lane, gb + 4 * lane);
        if (lane == 0 && nb > 32) cp_async16(buf + kHalfStage + 128, gb + 128);
      }
      return m;
    }
    {
      // crosses piece ends: each lane stages its own real tokens with 4-byte
      // copies (the store looks the pieces up again and reads them back)
      m.kind = 2;
      const uint32_t tp = t0 + 4u * lane;
      const int32_t last = P.used - 1;
      int32_t t = min((int32_t)tp, last);
      int32_t qi = P.find_lane(t);
      Piece q = P.get(qi);
#pragma unroll
      for (int e = 0; e < 4; e++) {
        t = min((int32_t)tp + e, last);
        const bool same = t < q.end;
        if (!__all_sync(0xffffffffu, same)) {
          const Piece nq = P.get(same ? qi : qi + 1);
          if (!same) {
            q = nq;
            qi++;
          }
        }
        if ((int32_t)tp + e <= last && tp < p.T)
          cp_async4(buf + 4 * lane + e, p.tokens + q.src + (t - q.start));
      }
    }
  }
  return m;
}

template <class PV>
__device__ __forceinline__ void tile_store(const GatherParams &p, const PV &P, uint32_t t0,
                                           int lane, size_t obase, const int32_t *buf,
                                           const TileMeta &mref, uint64_t &acc, int &learned) {
  const TileMeta m = mref;
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
    dc = make_int4(m.doc, m.doc, m.doc, m.doc);
    const int32_t th = m.mthr;
    mk = (x >= th ? 1u : 0u) | (x + 1 >= th ? 1u << 8 : 0u) | (x + 2 >= th ? 1u << 16 : 0u) |
         (x + 3 >= th ? 1u << 24 : 0u);
  } else if (m.kind == 3) {
    // at most two pieces: position i of the tile reads run a (i < bnd) or run
    // b, then padding from nreal on
    int32_t e0[4], e1[4], e2[4];
#pragma unroll
    for (int e = 0; e < 4; e++) {
      // selects, not branches: the lanes around the boundary do not diverge
      const int32_t i = 4 * lane + e;
      const bool in_a = i < m.bnd, real = i < m.nreal;
      const int32_t x = in_a ? m.x0 + i : i - m.bnd;
      const int32_t w = in_a ? m.sh + i : kHalfStage + m.sh2 + x;
      const int32_t v = buf[real ? w : 0];
      e0[e] = real ? v : p.pad_id;
      e1[e] = real ? x : 0;
      e2[e] = real ? (in_a ? m.doc : m.doc2) : -1;
      if (real && x >= (in_a ? m.mthr : m.mthr2)) mk |= 1u << (8 * e);
    }
    tk = make_int4(e0[0], e0[1], e0[2], e0[3]);
    ps = make_int4(e1[0], e1[1], e1[2], e1[3]);
    dc = make_int4(e2[0], e2[1], e2[2], e2[3]);
  } else {
    // every lane looks its four positions up together (the lookups shuffle);
    // positions past the window's end become padding afterwards
    int32_t e0[4], e1[4], e2[4];
    const int32_t last = P.used - 1;
    int32_t t = min((int32_t)tp, last);
    int32_t qi = P.find_lane(t);
    Piece pc = P.get(qi);
#pragma unroll
    for (int e = 0; e < 4; e++) {
      t = min((int32_t)tp + e, last);
      const bool same = t < pc.end;
      if (!__all_sync(0xffffffffu, same)) {
        // positions rise one at a time and no piece of a window is empty:
        // one past a piece's end is the next piece's start
        const Piece nq = P.get(same ? qi : qi + 1);
        if (!same) {
          pc = nq;
          qi++;
        }
      }
      const int32_t x = t - pc.start;
      const bool real = (int32_t)tp + e <= last && tp < p.T;
      e0[e] = real ? buf[4 * lane + e] : p.pad_id;
      e1[e] = real ? x : 0;
      e2[e] = real ? pc.doc : -1;
      if (real && x >= pc.mthr) mk |= 1u << (8 * e);
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
  // an all-padding tile's terms come from the context's table of padding
  // sums (added once per row by the last warp)
  if (m.kind == 0) return;
  acc += fp_term(tk.x, ps.x, dc.x, mk & 1u, tp);
  acc += fp_term(tk.y, ps.y, dc.y, (mk >> 8) & 1u, tp + 1);
  acc += fp_term(tk.z, ps.z, dc.z, (mk >> 16) & 1u, tp + 2);
  acc += fp_term(tk.w, ps.w, dc.w, (mk >> 24) & 1u, tp + 3);
  learned += __popc(mk);
}

// This warp's tiles: t0 = warp * 128 + m * 1024, through a ring of kStages
// shared-memory buffers filled by cp.async; each tile's description waits in
// shared memory beside its buffer (written by lane 0, read after __syncwarp).
template <int W, class PV>
__device__ __forceinline__ void warp_tiles(const GatherParams &p, const PV &P, int warp, int lane,
                                           size_t obase, int32_t (*ring)[stage_words<W>()],
                                           TileMeta *meta, uint64_t &acc, int &learned) {
  constexpr uint32_t kStride = W * kTile;
  const uint32_t first = (uint32_t)warp * kTile;
  const int n_tiles = first < p.T ? (int)((p.T - first + kStride - 1) / kStride) : 0;
#pragma unroll
  for (int m = 0; m < kStages - 1; m++) {
    if (m < n_tiles) {
      const TileMeta t = tile_issue<(W <= 8)>(p, P, first + m * kStride, lane, ring[m]);
      if (lane == 0) meta[m] = t;
    }
    cp_async_commit();
  }
#pragma unroll 1
  for (int mm = 0; mm < n_tiles; mm++) {
    const int mi = mm + kStages - 1;
    const int slot_i = mi % kStages;
    if (mi < n_tiles) {
      const TileMeta t = tile_issue<(W <= 8)>(p, P, first + mi * kStride, lane, ring[slot_i]);
      if (lane == 0) meta[slot_i] = t;
    }
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const int slot = mm % kStages;
    tile_store(p, P, first + mm * kStride, lane, obase, ring[slot], meta[slot], acc, learned);
    __syncwarp();
  }
}

// W warps per row: 4 (ten rows per SM) for rows up to 8192 positions, 8 (five
// rows) up to 16384, 16 (two rows) beyond: long rows come fewer to a launch,
// so each is given more warps.
template <int W>
__global__ void __launch_bounds__(W * 32, 40 / W)
    gather_kernel(const GatherParams p) {
  __shared__ __align__(16) int32_t s_tok[W][kStages][stage_words<W>()];
  __shared__ TileMeta s_meta[W][kStages];
  __shared__ unsigned long long s_acc;
  __shared__ int s_learned;
  __shared__ int s_done;

  const uint32_t blk = blockIdx.x;
  const uint32_t step_local = blk / p.n_rows;
  const uint32_t row_local = blk - step_local * p.n_rows;
  const uint32_t k = p.step0 + step_local;
  const uint32_t i = p.row0 + row_local;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    s_acc = 0;
    s_learned = 0;
    s_done = 0;
  }
  __syncthreads();

  // the row's window: pieces [ws, we) of the context's piece table, from
  // token `clip` of the first (wrap packing; 0 for greedy windows)
  const int4 win = p.row_win[(size_t)k * p.B + i];
  int64_t ws = win.x, we = win.y;
  int32_t clip = win.z;
  if (ws < 0 || we < ws) ws = we = clip = 0;  // a row past the end of its stream: all padding
  const int32_t np = (int32_t)(we - ws);
  const int64_t sbase = __ldg(p.node_S + ws) + clip;
  const int64_t used64 = min(__ldg(p.node_S + we) - sbase, (int64_t)p.T);
  int32_t used = (int32_t)used64;
  if (used64 < 0 || clip < 0 || (np == 0 && clip != 0)) {
    set_error(p.err, kDevBadNode);
    used = 0;
  }

  const size_t obase = (size_t)blk * p.T;
  uint64_t acc = 0;
  int learned = 0;
  if (np <= 32) {
    WarpPieces P;
    P.np = np;
    P.used = used;
    P.S = INT_MAX;
    P.src = 0;
    P.doc = -1;
    P.mthr = 0;
    if (lane < np) {
      P.S = lane == 0 ? 0 : (int32_t)(__ldg(p.node_S + ws + lane) - sbase);
      P.src = __ldg(p.node_src + ws + lane) + (lane == 0 ? clip : 0);
      P.doc = __ldg(p.node_doc + ws + lane);
      P.mthr = __ldg(p.node_mthr + ws + lane);
      if (lane == 0) P.mthr = clip_threshold(P.mthr, clip);
    }
    warp_tiles<W>(p, P, warp, lane, obase, s_tok[warp], s_meta[warp], acc, learned);
  } else {
    TablePieces P;
    P.S = p.node_S + ws;
    P.srcs = p.node_src + ws;
    P.docs = p.node_doc + ws;
    P.mthrs = p.node_mthr + ws;
    P.sbase = sbase;
    P.np = np;
    P.used = used;
    P.clip = clip;
    warp_tiles<W>(p, P, warp, lane, obase, s_tok[warp], s_meta[warp], acc, learned);
  }

  // combine the warps' sums; the last warp to arrive writes the row's values
  acc = warp_sum_u64(acc);
  learned = warp_sum_i32(learned);
  if (lane == 0) {
    atomicAdd(&s_acc, (unsigned long long)acc);
    atomicAdd(&s_learned, learned);
    __threadfence_block();
    if (atomicAdd(&s_done, 1) == W - 1) {
      __threadfence_block();
      // tiles from the first one at or after `used` are all padding
      const uint64_t a = *reinterpret_cast<volatile unsigned long long *>(&s_acc) +
                         __ldg(p.pad_tail + ((uint32_t)used + kTile - 1) / kTile);
      p.row_fp[blk] = splitmix64(a);
      p.row_learned[blk] = *reinterpret_cast<volatile int *>(&s_learned);
      if (p.row_len) {
        // real positions come first; report them rounded up to the bucket
        const uint64_t b = p.len_bucket;
        const uint64_t len = b ? min((((uint64_t)used + b - 1) / b) * b, (uint64_t)p.T) : used;
        p.row_len[blk] = (int32_t)len;
      }
    }
  }
}

// Batch fingerprint of each update: F = splitmix64(F ^ fp_i) over its rows,
// in row order.  One block per update stages the row values in shared memory
// so the serial fold never waits on global memory.
constexpr int kFoldChunk = 2048;

__global__ void __launch_bounds__(256)
    batch_fp_kernel(const uint64_t *__restrict__ row_fp, uint32_t n_rows,
                    uint64_t *__restrict__ out) {
  pdl_wait_then_release();
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

// Padding sums per tile: tile k (positions [128k, min(128k + 128, T))) of
// a row of padding; then suffix sums, pad_tail[k] = the terms of positions
// [128k, T), pad_tail[n_tiles] = 0.
__global__ void __launch_bounds__(256)
    pad_tiles_kernel(int32_t pad_id, uint32_t T, uint32_t n_tiles, uint64_t *__restrict__ tile) {
  pdl_wait_then_release();
  const uint32_t k = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (k >= n_tiles) return;
  uint64_t acc = 0;
#pragma unroll
  for (int e = 0; e < 4; e++) {
    const uint32_t t = k * kTile + 4 * lane + e;
    if (t < T) acc += fp_term(pad_id, 0, -1, 0u, t);
  }
  acc = warp_sum_u64(acc);
  if (lane == 0) tile[k] = acc;
}

__global__ void __launch_bounds__(1024)
    pad_suffix_kernel(const uint64_t *__restrict__ tile, uint32_t n_tiles,
                      uint64_t *__restrict__ pad_tail) {
  pdl_wait_then_release();
  __shared__ uint64_t s_w[32];
  __shared__ uint64_t s_carry;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_carry = 0;
    pad_tail[n_tiles] = 0;
  }
  __syncthreads();
  // chunks of 1024 tiles from the end: suffix sum = carry + inclusive sum of
  // the reversed chunk
  for (uint32_t c0 = 0; c0 < n_tiles; c0 += 1024) {
    const uint32_t r = c0 + threadIdx.x;                // reversed index
    const uint64_t v = r < n_tiles ? tile[n_tiles - 1 - r] : 0;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_w[w] = x;
    __syncthreads();
    if (w == 0) {
      uint64_t z = s_w[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, z, o);
        if (lane >= o) z += y;
      }
      s_w[lane] = z;
    }
    __syncthreads();
    const uint64_t incl = s_carry + (w ? s_w[w - 1] : 0) + x;
    if (r < n_tiles) pad_tail[n_tiles - 1 - r] = incl;
    __syncthreads();
    if (threadIdx.x == 0) s_carry += s_w[31];
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_pad_tail(int32_t pad_id, uint32_t T, uint64_t *tile_scratch,
                            uint64_t *pad_tail, cudaStream_t st) {
  const uint32_t n_tiles = (T + kTile - 1) / kTile;
  ++launch_counter();
  pdl_launch(pad_tiles_kernel, (n_tiles * 32 + 255) / 256, 256, 0, st, pad_id, T, n_tiles, tile_scratch);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++launch_counter();
  pdl_launch(pad_suffix_kernel, 1, 1024, 0, st, tile_scratch, n_tiles, pad_tail);
  return cudaGetLastError();
}

cudaError_t launch_gather(const GatherParams &p, cudaStream_t st) {
  const uint64_t n = (uint64_t)p.n_steps * p.n_rows;
  if (n == 0) return cudaSuccess;
  ++launch_counter();
  if (p.T <= 8192)
    gather_kernel<4><<<(unsigned)n, 4 * 32, 0, st>>>(p);
  else if (p.T <= 16384)
    gather_kernel<8><<<(unsigned)n, 8 * 32, 0, st>>>(p);
  else
    gather_kernel<16><<<(unsigned)n, 16 * 32, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_batch_fp(const uint64_t *row_fp, uint32_t n_steps, uint32_t n_rows,
                            uint64_t *out, cudaStream_t st) {
  ++launch_counter();
  pdl_launch(batch_fp_kernel, n_steps, 256, 0, st, row_fp, n_rows, out);
  return cudaGetLastError();
}

}  // namespace nsk
