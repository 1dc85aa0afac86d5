// Host-side launchers of the library's kernels (internal interface between
// the C ABI in api.cu and the kernels in init_kernels.cu / gather.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace nsk {

// Kernels launched by this thread so far (each launcher adds its own).
uint64_t &launch_counter();

// A launch over per-stream segments: stream j owns items [0, count_j), laid
// out in blocks of `block` items; blk_base[j] is the first block of stream j
// (host-computed prefix, J + 1 entries, on the device).
struct SegGrid {
  const uint32_t *blk_base;  // [J + 1]
  uint32_t J;
  uint32_t n_blocks;
};

// ---- validation, keys, quotas ---------------------------------------------
cudaError_t launch_validate_offsets(const int64_t *offs, uint32_t n_docs, uint64_t n_tokens,
                                    int *err, int n_sms, cudaStream_t st);
// The shuffle's round keys of every stream (keys[4 j + r]); with est_tok
// (per stream, the recipe's estimate of the tokens its windows hold) also
// pos_lim[j], the shuffled positions taken of stream j (about those its
// estimate needs for a stream without a held-out rate, all for the others).
cudaError_t launch_keys_bound(uint64_t seed, uint32_t J, uint64_t *keys, const uint32_t *sdb,
                              const int64_t *offs, const uint16_t *stream_bp,
                              const unsigned long long *est_tok, uint32_t *pos_lim,
                              cudaStream_t st);
// The schedule on the device: piece p covers updates [begin[p], begin[p+1])
// (the last one up to K) with B[p] rows per update and weights sw[p][S],
// tw[p][J]; a recipe without a schedule is one piece.
struct QuotaPieces {
  const uint32_t *begin;
  const uint32_t *B;
  const uint32_t *sw;
  const uint32_t *tw;
  uint32_t P;
};
cudaError_t launch_quota_sources(QuotaPieces q, uint32_t S, uint32_t K, int32_t *src_quota,
                                 cudaStream_t st);
// Every quota block adds 1 to *ready (if not null) once its streams' last
// table row is written.
cudaError_t launch_quota_strata(QuotaPieces q, const int32_t *src_quota,
                                const uint32_t *src_first, uint32_t S, uint32_t J, uint32_t K,
                                uint32_t max_strata, int32_t *quota, int32_t *cum,
                                unsigned *ready, cudaStream_t st);
// Both levels in one kernel when n_sources <= 32 and every source has <= 32 strata.
cudaError_t launch_quota_warp(QuotaPieces q, uint32_t S, const uint32_t *src_first, uint32_t J,
                              uint32_t K, uint32_t max_strata, int32_t *quota, int32_t *cum,
                              unsigned *ready, cudaStream_t st);
cudaError_t launch_row_base(const int32_t *quota, uint32_t J, uint32_t K, int32_t *rb,
                            cudaStream_t st);

// ---- held-out hash, order, scans ------------------------------------------
// stream_bp_heldout_mode: null for the training stream; for the validation
// stream the per-stream rates (a stream of a source that holds nothing out
// keeps nothing)
// pos_lim (per stream, or NULL: every position): the shuffled positions
// taken, from launch_keys_bound; of the others, those a scan tile that is
// not skipped reads get length 0 (launch_scan_pieces)
cudaError_t launch_order(SegGrid g, const uint32_t *sdb, const uint64_t *keys,
                         const int64_t *offs, uint64_t n_tokens, uint32_t D0,
                         const uint16_t *stream_bp_heldout_mode, const uint32_t *pos_lim,
                         uint32_t *order, uint32_t *klen, int *err, int n_sms,
                         cudaStream_t st);
// held-out documents of the prefix each stream's horizon reaches get klen 0
// copy_dst non-null: tokens is host memory the device can address, and
// every hashed document is also written to copy_dst (tokens_read counts them).
// hashed[0] and hashed[1] count the tokens and the documents hashed.
// pre_cap (per stream kept tokens, or NULL): where a stream stops before the
// quota table is known.  frontier and prog (per stream, zeroed before the
// first round, carried into the second): the next position to grab, and the
// progress word (decided kept tokens plus estimates of the grabs in flight,
// in bits 16 and up; the grabs in flight below).  The grid is n_sms times the
// hash's CTAs per SM: fewer than 2^16 warps, so the word's count cannot wrap
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
                               int n_sms, cudaStream_t st);
// A stream whose windows needed are fewer than this keeps the full bound in
// the hash's second round (its sample would be too small to measure a fill).
constexpr int64_t kSpeculateMinWindows = 256;
// need_num: the fraction (of 1024) of each stream's bound the second hash
// round stops at, from its measured packing fill (first_num: the first
// round's)
cudaError_t launch_fill_need(const uint32_t *sdb, uint32_t J, uint32_t D0,
                             const uint16_t *stream_bp, const uint32_t *order, const uint32_t *klen,
                             const int64_t *offs, uint64_t n_tokens, const int32_t *cum_last,
                             uint32_t T, uint32_t G, uint32_t first_num,
                             const unsigned long long *pre_cap, uint16_t *need_num,
                             cudaStream_t st);
// The kept tokens of positions [0, cutoff[j]) of every stream with
// stream_bp[j] == 0, copied from src (host memory the device can address) to
// dst; the grid has a block per 8 chunks of copy_chunk_tokens() kept tokens
// of those prefixes.
cudaError_t launch_copy_prefix(SegGrid g, const uint32_t *sdb, uint32_t D0,
                               const uint32_t *cutoff, const uint16_t *stream_bp,
                               const uint32_t *order, const uint32_t *klen, const int64_t *kex,
                               const int64_t *offs, const int32_t *src, int32_t *dst,
                               unsigned long long *tokens_read, cudaStream_t st);
uint32_t copy_chunk_tokens();
// kex[i] = sum_{i' < i} klen[i'], pex[i] = sum_{i' < i} ceil(klen[i'] / T), i in [0, n].
// pos_lim (per stream, or NULL): streams shuffled only in part, whose
// positions past b_j + pos_lim_j have length 0 (written there by the
// shuffle only where a scan tile reaches into the shuffled part or the next
// stream: the other tiles are skipped); there kex and pex are written only
// where a tile of the scan reaches into the shuffled part or the next stream
// (the cutoff reads them up to b_j + pos_lim_j and at stream ends).  *done:
// zeroed before.
cudaError_t launch_scan_pieces(const uint32_t *klen, uint64_t n, uint32_t T, int64_t *kex,
                               int64_t *pex, void *scratch, size_t scratch_bytes,
                               const uint32_t *sdb, uint32_t J, uint32_t D0,
                               const uint32_t *pos_lim, unsigned *done, int n_sms,
                               cudaStream_t st);
size_t scan_scratch_bytes(uint64_t n);
// per stream: cutoff c_j, pieces and kept tokens before it (rmax given as
// cum_last, the quota table's last row); then node_base[j] (J + 1 entries:
// the first node of each stream, one terminal node after each), and the
// words the host reads back besides: cum_last[j] at rb[rb_rmax + j], the
// error word at rb[rb_err].  *done: zeroed before.
cudaError_t launch_cutoff(const uint32_t *sdb, uint32_t J, uint32_t D0, const int64_t *kex,
                          const int64_t *pex, const int32_t *cum_last, uint32_t T, uint32_t G,
                          const uint16_t *need_num, const uint32_t *pos_lim, uint32_t *cutoff,
                          int64_t *npieces, int64_t *ptokens, int64_t *node_base, uint32_t *rb,
                          uint32_t rb_rmax, uint32_t rb_err, const int *err, unsigned *done,
                          cudaStream_t st);

// ---- pieces, next, jump tables, windows -----------------------------------
cudaError_t launch_expand(SegGrid g, const uint32_t *sdb, uint32_t D0, const uint32_t *cutoff,
                          const uint32_t *order, const uint32_t *klen, const int64_t *kex,
                          const int64_t *pex, const int64_t *node_base, const int64_t *npieces,
                          const int64_t *offs, const int32_t *loss_start, uint32_t T,
                          int64_t *node_src, int32_t *node_doc, int32_t *node_mthr,
                          int64_t *node_S, cudaStream_t st);
cudaError_t launch_next(SegGrid g, const int64_t *node_base, const int64_t *npieces,
                        const int64_t *node_S, uint32_t T, int32_t *next, cudaStream_t st);
cudaError_t launch_jump_level(const int32_t *up_prev, int64_t n_nodes, int32_t *up_next,
                              cudaStream_t st);
// levels l and l + 1 from level l - 1 in one launch
cudaError_t launch_jump_two_levels(const int32_t *up_prev, int64_t n_nodes, int32_t *up_next,
                                   int32_t *up_next2, cudaStream_t st);
// positions a thread of the shuffle kernel takes (its grid: blocks of 256
// threads over segments of 256 * order_positions_per_thread() positions)
uint32_t order_positions_per_thread();
// levels: [n_levels][n_nodes], level l maps a node to the node 2^l windows on
cudaError_t launch_count_windows(const int32_t *levels, int64_t n_nodes, uint32_t n_levels,
                                 const int64_t *node_base, const int64_t *npieces, uint32_t J,
                                 uint32_t *W, cudaStream_t st);
cudaError_t launch_window_starts(SegGrid g, const int32_t *levels, int64_t n_nodes,
                                 uint32_t n_levels, const int64_t *node_base, const uint32_t *W,
                                 const int64_t *wbase, int32_t *win_start, cudaStream_t st);
// row_win[k][i] = (first piece, end piece, clip, 0) of the window slot i of
// update k takes, or (-1, -1) when the row lies past the end of its stream
// (win_end / win_clip: wrap packing's tables; null for greedy windows); G > 0
// reads windows in a shuffled order within segments, shuffle_rows shuffles the
// rows of every update.  In the same launch: *bad_inv (zeroed before) = K - k
// for the first update k that asks a stream for a window it does not have
// (0 if none), then the valid horizon *valid (through that update with
// drain, else before it) and ubase[j] (J + 1 entries: the first digest item
// of each stream's used windows).  *done: zeroed before.
cudaError_t launch_row_table(const int32_t *rb, const int32_t *cum, const uint32_t *W,
                             const int64_t *wbase, const int32_t *win_start, const int32_t *next,
                             const int32_t *win_end, const int32_t *win_clip, uint32_t J,
                             uint32_t B, uint32_t K, uint64_t seed, uint32_t G,
                             uint32_t shuffle_rows, int4 *row_win, int *err, uint32_t *bad_inv,
                             uint32_t drain, uint32_t *valid, int64_t *ubase, unsigned *done,
                             cudaStream_t st);
// Wrap packing: windows of exactly T tokens of each stream's kept run.
cudaError_t launch_wrap_windows(SegGrid g, const int64_t *node_base, const int64_t *npieces,
                                const int64_t *node_S, const uint32_t *cutoff,
                                const uint32_t *sdb, uint32_t J, uint32_t T, uint32_t *W,
                                const int64_t *wbase, int32_t *win_start, int32_t *win_end,
                                int32_t *win_clip, cudaStream_t st);

// ---- order digest ---------------------------------------------------------
constexpr int kDigestScalars = 12;
struct DigestHeader {
  uint64_t scalars[kDigestScalars];  // T, B, K, valid, flags, pad, seed, key, S, J, G, bucket
  const uint32_t *source_weight;  // [S]
  const uint16_t *source_bp;      // [S]
  const uint32_t *sdb;            // [J + 1]
  const uint32_t *ssrc;           // [J]
  const uint32_t *tw;             // [J]
  const uint64_t *piece_items;    // the schedule's items (none without one)
  uint64_t n_piece_items;
  uint32_t S, J;
};
// The order digest over the valid horizon (*valid and ubase from
// launch_row_table) into *digest; in the same launch each stream's window
// count W[j] is copied to rb[rb_W + j] and the error word to rb[rb_err].
// acc[0] and *done: zeroed before.
cudaError_t launch_digest(const DigestHeader &h, const int32_t *quota, uint32_t K, SegGrid wg,
                          const int64_t *wbase, const int32_t *win_start,
                          const int64_t *node_src, const int32_t *node_doc, const int64_t *offs,
                          const uint32_t *valid, const int64_t *ubase, const uint32_t *W,
                          uint64_t seed, uint32_t G, const int32_t *win_clip, int *err,
                          unsigned long long *acc, uint64_t *digest, uint32_t *rb, uint32_t rb_W,
                          uint32_t rb_err, unsigned *done, cudaStream_t st);

// ---- per-step assembly ----------------------------------------------------
struct GatherParams {
  // corpus
  const int32_t *tokens;
  // context tables
  const int4 *row_win;      // [K][B]: pieces [x, y) of the row's window from offset z of
                            // the first; x < 0 past the end
  const int64_t *node_S;    // [nodes]
  const int64_t *node_src;  // [nodes]
  const int32_t *node_doc;  // [nodes]
  const int32_t *node_mthr; // [nodes]
  int *err;
  // launch
  uint32_t B, T, step0, n_steps, row0, n_rows;
  int32_t pad_id;
  // outputs
  int32_t *tokens_out, *pos_out, *doc_out;
  uint8_t *mask_out;
  uint64_t *row_fp;
  int32_t *row_learned;
  int32_t *row_len;         // [n_steps][rows] or null
  uint32_t len_bucket;
  const uint64_t *pad_tail;  // [T/128 + 1]: fingerprint terms of padding from tile k on
};
cudaError_t launch_gather(const GatherParams &p, cudaStream_t st);
// pad_tail[k] = the sum of the fingerprint terms of a padding row's positions
// [128k, T); tile_scratch holds ceil(T / 128) words.
cudaError_t launch_pad_tail(int32_t pad_id, uint32_t T, uint64_t *tile_scratch,
                            uint64_t *pad_tail, cudaStream_t st);
// out[s] = sum of row_learned[s * n_rows .. (s + 1) * n_rows) (learned.cu)
cudaError_t launch_step_learned(const int32_t *row_learned, uint32_t n_steps, uint32_t n_rows,
                                int64_t *out, cudaStream_t st);
cudaError_t launch_batch_fp(const uint64_t *row_fp, uint32_t n_steps, uint32_t n_rows,
                            uint64_t *out, cudaStream_t st);

}  // namespace nsk
