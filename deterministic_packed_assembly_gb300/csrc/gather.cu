// Per-update assembly: one CTA per (update, row).  The row's stream and
// window come from the quota tables; the window's pieces are copied in order
// into T positions of tokens / position ids / document ids / loss mask, the
// rest padded; the row's fingerprint and learned-position count are reduced
// in the same pass.
//
// Rows of exactly T positions, padded (Linnet training docs, Supervised
// fine-tuning); a position id of 0 starts each sequence within a row (Other
// trainers); only completion tokens are learned (Supervised fine-tuning);
// rows are a pure function of (recipe, seed, update, row), so any split of
// the rows gives the same bytes ("Zephon: deterministic data loading",
// checkpoint on 16 GPUs, resume on 8/32/64).
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace nsk {

namespace {

constexpr int kGatherWarps = 8;
constexpr int kTile = 128;  // positions per warp per round: 32 lanes x 4

// Fingerprint terms and learned count of four consecutive positions t0..t0+3:
// key_t = a_t ^ ((b_t | t << 40) * golden), a_t = (u32 tok << 32) | u32 doc,
// b_t = (mask << 32) | u32 pos.
__device__ __forceinline__ void fingerprint4(uint64_t &acc, int &learned, const int4 &tk,
                                             const int4 &ps, const int4 &dc, uint32_t mk,
                                             uint32_t t0) {
  const int32_t tok[4] = {tk.x, tk.y, tk.z, tk.w};
  const int32_t pos[4] = {ps.x, ps.y, ps.z, ps.w};
  const int32_t doc[4] = {dc.x, dc.y, dc.z, dc.w};
#pragma unroll
  for (int e = 0; e < 4; e++) {
    const uint64_t m = (mk >> (8 * e)) & 1u;
    const uint64_t a = ((uint64_t)(uint32_t)tok[e] << 32) | (uint64_t)(uint32_t)doc[e];
    const uint64_t b = (m << 32) | (uint64_t)(uint32_t)pos[e];
    const uint64_t key = a ^ ((b | ((uint64_t)(t0 + e) << 40)) * kGolden);
    acc += splitmix64(key);
  }
  learned += __popc(mk);
}

__device__ __forceinline__ int4 shfl_down4(const int4 &v) {
  int4 r;
  r.x = __shfl_down_sync(0xffffffffu, v.x, 1);
  r.y = __shfl_down_sync(0xffffffffu, v.y, 1);
  r.z = __shfl_down_sync(0xffffffffu, v.z, 1);
  r.w = __shfl_down_sync(0xffffffffu, v.w, 1);
  return r;
}

__global__ void __launch_bounds__(kGatherWarps * 32)
    gather_kernel(const GatherParams p) {
  __shared__ int64_t s_ws, s_we, s_sbase;
  __shared__ int32_t s_used;
  __shared__ uint64_t s_fp[kGatherWarps];
  __shared__ int s_learned[kGatherWarps];

  const uint32_t blk = blockIdx.x;
  const uint32_t step_local = blk / p.n_rows;
  const uint32_t row_local = blk - step_local * p.n_rows;
  const uint32_t k = p.step0 + step_local;
  const uint32_t i = p.row0 + row_local;
  const uint32_t T = p.T;

  if (threadIdx.x == 0) {
    const int32_t *rbk = p.rb + (size_t)k * (p.J + 1);
    const int64_t j = last_le<int32_t, int64_t>(rbk, 0, (int64_t)p.J, (int32_t)i);
    const int64_t r = (int64_t)p.cum[(size_t)k * p.J + j] + ((int64_t)i - rbk[j]);
    int64_t ws = 0, we = 0, sbase = 0;
    int64_t used = 0;
    if (r < (int64_t)p.W[j]) {
      ws = p.win_start[p.wbase[j] + r];
      if (ws >= 0) {
        we = p.next[ws];
        sbase = p.node_S[ws];
        used = p.node_S[we] - sbase;
      }
      if (ws < 0 || we <= ws || used <= 0 || used > (int64_t)T) {
        set_error(p.err, kDevBadNode);
        ws = we = sbase = 0;
        used = 0;
      }
    }
    s_ws = ws;
    s_we = we;
    s_sbase = sbase;
    s_used = (int32_t)used;
  }
  __syncthreads();
  const int64_t ws = s_ws, we = s_we, sbase = s_sbase;
  const int32_t used = s_used;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t obase = (size_t)blk * T;
  uint64_t acc = 0;
  int learned = 0;

  for (uint32_t t0 = (uint32_t)warp * kTile; t0 < T; t0 += kGatherWarps * kTile) {
    const uint32_t tp = t0 + 4u * lane;
    int4 tk, ps, dc;
    uint32_t mk = 0;
    if ((int32_t)t0 >= used) {
      tk = make_int4(p.pad_id, p.pad_id, p.pad_id, p.pad_id);
      ps = make_int4(0, 0, 0, 0);
      dc = make_int4(-1, -1, -1, -1);
    } else {
      // the piece holding the tile's first position
      const int64_t q = last_le<int64_t, int64_t>(p.node_S, ws, we, sbase + (int64_t)t0);
      const int64_t qs = __ldg(p.node_S + q) - sbase;
      const int64_t qe = __ldg(p.node_S + q + 1) - sbase;
      if (qe >= (int64_t)t0 + kTile) {
        // the whole tile lies in piece q: one realigned 16-byte load per lane
        const int64_t x0 = (int64_t)t0 - qs;
        const int64_t srcw = __ldg(p.node_src + q) + x0;
        const int sh = (int)(srcw & 3);
        const int4 *src4 = reinterpret_cast<const int4 *>(p.tokens + (srcw - sh));
        const int4 v = __ldg(src4 + lane);
        if (sh == 0) {
          tk = v;
        } else {
          int4 nv = shfl_down4(v);
          if (lane == 31) nv = __ldg(src4 + 32);
          if (sh == 1)
            tk = make_int4(v.y, v.z, v.w, nv.x);
          else if (sh == 2)
            tk = make_int4(v.z, v.w, nv.x, nv.y);
          else
            tk = make_int4(v.w, nv.x, nv.y, nv.z);
        }
        const int32_t x = (int32_t)x0 + 4 * lane;
        ps = make_int4(x, x + 1, x + 2, x + 3);
        const int32_t d = __ldg(p.node_doc + q);
        dc = make_int4(d, d, d, d);
        const int32_t th = __ldg(p.node_mthr + q);
        mk = (x >= th ? 1u : 0u) | (x + 1 >= th ? 1u << 8 : 0u) | (x + 2 >= th ? 1u << 16 : 0u) |
             (x + 3 >= th ? 1u << 24 : 0u);
      } else if (tp < T) {
        // the tile crosses piece ends: each lane finds its pieces
        int32_t tkv[4], psv[4], dcv[4];
        int64_t qq = -1, qqs = 0, qqe = 0;
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int32_t t = (int32_t)tp + e;
          if (t >= used) {
            tkv[e] = p.pad_id;
            psv[e] = 0;
            dcv[e] = -1;
            continue;
          }
          if (qq < 0) {
            qq = last_le<int64_t, int64_t>(p.node_S, q, we, sbase + (int64_t)t);
            qqs = __ldg(p.node_S + qq) - sbase;
            qqe = __ldg(p.node_S + qq + 1) - sbase;
          }
          while ((int64_t)t >= qqe) {
            qq++;
            qqs = qqe;
            qqe = __ldg(p.node_S + qq + 1) - sbase;
          }
          const int32_t x = t - (int32_t)qqs;
          tkv[e] = __ldg(p.tokens + __ldg(p.node_src + qq) + x);
          psv[e] = x;
          dcv[e] = __ldg(p.node_doc + qq);
          if (x >= __ldg(p.node_mthr + qq)) mk |= 1u << (8 * e);
        }
        tk = make_int4(tkv[0], tkv[1], tkv[2], tkv[3]);
        ps = make_int4(psv[0], psv[1], psv[2], psv[3]);
        dc = make_int4(dcv[0], dcv[1], dcv[2], dcv[3]);
      }
    }
    if (tp < T) {
      __stcs(reinterpret_cast<int4 *>(p.tokens_out + obase + tp), tk);
      __stcs(reinterpret_cast<int4 *>(p.pos_out + obase + tp), ps);
      __stcs(reinterpret_cast<int4 *>(p.doc_out + obase + tp), dc);
      __stcs(reinterpret_cast<unsigned int *>(p.mask_out + obase + tp), mk);
      fingerprint4(acc, learned, tk, ps, dc, mk, tp);
    }
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

// Batch fingerprint of each update: F = splitmix64(F ^ fp_i) over its rows.
__global__ void batch_fp_kernel(const uint64_t *__restrict__ row_fp, uint32_t n_steps,
                                uint32_t n_rows, uint64_t *__restrict__ out) {
  const uint32_t s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n_steps) return;
  const uint64_t *f = row_fp + (size_t)s * n_rows;
  uint64_t F = 0;
  for (uint32_t i = 0; i < n_rows; i++) F = splitmix64(F ^ f[i]);
  out[s] = F;
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
  batch_fp_kernel<<<(n_steps + 63) / 64, 64, 0, st>>>(row_fp, n_steps, n_rows, out);
  return cudaGetLastError();
}

}  // namespace nsk
