/*
 * nspack.h -- C ABI of the GB300 library for deterministic packed assembly.
 *
 * Pre-tokenized documents from a weighted mixture of sources become fixed
 * [B, T] global batches (tokens, position ids, document ids, loss masks) plus
 * a 64-bit fingerprint and a learned-position count per row.  A batch depends
 * only on the recipe, the seed and the update index, never on how its rows are
 * split between calls, devices or processes.
 *
 * What the operations compute, and where it is stated:
 *  - held-out split: 1 % of every source's documents (5 % for one source), by
 *    a hash of the document's content that no line's seed changes --
 *    NeuronSpark-Trainer README, Concepts;
 *  - shuffle: a file's documents are visited in a seed-keyed random order --
 *    same section;
 *  - mixture: in every update each source's window count is at most two
 *    off its recipe share, and each stratum of a source at its share -- same
 *    section;
 *  - packing: windows of exactly T positions, cut at document ends, padded at
 *    the end -- same section, and Linnet training docs, Supervised
 *    fine-tuning; a document longer than T is cut into T-chunks;
 *  - assembly: a position id of 0 starts a new sequence within a row (Linnet
 *    training docs, Other trainers); only completion tokens are learned and a
 *    step is weighed by its count of learned positions (Supervised
 *    fine-tuning); rows past the end of the data learn nothing (Reinforcement
 *    learning, JAX);
 *  - elastic determinism: every global batch is byte-identical whatever the
 *    number of GPUs -- "Zephon: deterministic data loading", checkpoint on 16
 *    GPUs, resume on 8/32/64;
 *  - max_epochs 1: running out of a source is an error, never another epoch --
 *    NeuronSpark-Trainer README, Concepts; a resume checks the sample order's
 *    digest -- same README, Training.
 *
 * Conventions for every entry point:
 *  - All integers are little-endian; u64 arithmetic wraps.
 *  - Every argument is checked on the host before anything is enqueued; a
 *    failing check returns a negative NS_ERR_* code and changes nothing.
 *  - Kernels never trap.  An inconsistency found on the device is recorded in
 *    the context's device error word and reported by the next call that
 *    synchronises (ns_pack_fingerprint, ns_pack_check).
 *  - The context is immutable after ns_pack_init returns, so ns_pack_step may
 *    run concurrently on different CUDA streams.
 */
#ifndef NSPACK_H
#define NSPACK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define NS_OK 0
#define NS_ERR_INVALID_ARG (-1) /* an argument or the recipe is out of range */
#define NS_ERR_CUDA (-2)        /* a CUDA runtime call failed */
#define NS_ERR_OOM (-3)         /* the allocator returned NULL */
#define NS_ERR_EXHAUSTED (-4)   /* a stream has no window left for this update */
#define NS_ERR_HORIZON (-5)     /* update index at or past max_steps */
#define NS_ERR_BAD_INPUT (-6)   /* doc_offsets malformed (found on the device) */
#define NS_ERR_DEVICE (-7)      /* a kernel recorded an inconsistency */

/* ---- flags -------------------------------------------------------------- */
/* Allow the first update that runs a stream dry: its rows past the stream's
 * last window are empty (pad, pos 0, doc -1, mask 0); later updates return
 * NS_ERR_EXHAUSTED. */
#define NS_PACK_DRAIN 1u
/* Pack the validation stream: the held-out documents of every stream instead
 * of the kept ones (NeuronSpark-Trainer README, Concepts: a source's
 * validation rows are drawn from the held-out documents of all its strata).
 * Same shuffle, packing,
 * quotas and assembly; a source with a held-out rate of 0 has no windows. */
#define NS_PACK_HELDOUT 2u
/* Shuffle the rows of every update: slot i holds the row that would otherwise
 * be row rho_k(i), rho_k a keyed permutation of [0, B) (seed + 2, update k). */
#define NS_PACK_SHUFFLE_ROWS 4u
/* Wrap packing: concatenate each stream's kept documents and cut the run into
 * windows of exactly T tokens, across document ends (the flat packing with
 * the wrap algorithm of the pipeline example in "Zephon: deterministic data
 * loading").  A
 * piece is a document's run inside one window and its position ids start at
 * 0; a stream's last window may be partial (padded), and it counts only once
 * the whole stream is inside the reachable prefix. */
#define NS_PACK_WRAP 8u
/* The corpus (tokens, doc_offsets, loss_start) is in host memory: the
 * context keeps its own device copy (kept with the tables and counted in
 * table_bytes), offsets and loss starts copied first.  Tokens in page-locked
 * memory the device can address (cudaHostAlloc, or cudaHostRegister; 16-byte
 * aligned) are read where they lie, and only the documents the horizon
 * reaches cross the host link: the held-out hash writes every document it
 * reads into the copy, and a copy kernel brings over the reachable prefix of
 * every stream whose source has no held-out rate.  Tokens in other host
 * memory are copied whole, in groups of whole streams on a second stream,
 * each group hashed as soon as its copy lands.  ns_pack_info reports the
 * bytes read (host_bytes); the host buffers may be released once
 * ns_pack_init returns. */
#define NS_PACK_HOST_CORPUS 16u
/* The free callback is stream-ordered on cuda_stream: memory it takes back is
 * reused only by work queued on that stream after the free (a stream-ordered
 * pool such as PyTorch's caching allocator).  ns_pack_free then releases the
 * tables without waiting for the stream, unless ns_pack_step ran on another
 * stream.  Needs alloc and free. */
#define NS_PACK_ORDERED_FREE 32u

/* ---- limits ------------------------------------------------------------- */
#define NS_MAX_T (1u << 24)          /* T must be a multiple of 16, at most this */
#define NS_MAX_SOURCES 1024u
#define NS_MAX_STRATA_PER_SOURCE 1024u
#define NS_MAX_STREAMS 65536u
#define NS_MAX_WINDOW_SEGMENT (1u << 24)
#define NS_MAX_TOKENS (1ull << 47)   /* n_tokens must be below this */

typedef struct ns_pack_ctx ns_pack_ctx;

/* Device memory for the context's tables.  Called only inside ns_pack_init
 * (allocations) and ns_pack_init / ns_pack_free (frees); NULL alloc means
 * cudaMalloc / cudaFree.  Returned pointers must be 256-byte aligned. */
typedef void *(*ns_alloc_fn)(size_t bytes, void *user);
typedef void (*ns_free_fn)(void *ptr, void *user);

typedef struct {
  /* Corpus, on the device, borrowed (must outlive the context); with
   * NS_PACK_HOST_CORPUS in host memory instead, copied.  Documents are
   * contiguous runs of tokens: document d is tokens[doc_offsets[d] ..
   * doc_offsets[d+1]).  On the device, tokens must be 16-byte aligned and
   * doc_offsets and loss_start aligned for their types (8 and 4 bytes), else
   * NS_ERR_INVALID_ARG. */
  const int32_t *tokens;
  uint64_t n_tokens;          /* < NS_MAX_TOKENS */
  const int64_t *doc_offsets; /* [n_docs + 1], nondecreasing, lengths < 2^31 */
  const int32_t *loss_start;  /* [n_docs] or NULL: a token at in-document
                                 offset o is learned iff o >= loss_start[d];
                                 NULL learns every token */
  uint32_t n_docs;            /* < 2^31 */
  uint32_t n_sources;         /* 1 .. NS_MAX_SOURCES */
  uint32_t n_streams;         /* 1 .. NS_MAX_STREAMS: (source, stratum) pairs */
  uint32_t T;                 /* window length, multiple of 16, <= NS_MAX_T */
  /* Recipe, on the host, copied by ns_pack_init. */
  const uint32_t *stream_doc_begin;  /* [n_streams + 1], nondecreasing, <= n_docs:
                                        stream j owns documents [b[j], b[j+1]) */
  const uint32_t *stream_source;     /* [n_streams], nondecreasing, < n_sources;
                                        every source owns >= 1 stream */
  const uint32_t *source_weight;     /* [n_sources], > 0 */
  const uint32_t *stream_weight;     /* [n_streams], > 0, relative within its source */
  const uint16_t *source_heldout_bp; /* [n_sources], 0 .. 10000 basis points */
  uint64_t seed;     /* keys the shuffle */
  uint64_t hash_key; /* keys the held-out hash (not the seed, so every line agrees) */
  uint32_t B;        /* rows per update (global batch), >= 1 */
  uint32_t max_steps; /* horizon of the quota tables; max_steps * B < 2^31 */
  uint32_t flags;    /* NS_PACK_DRAIN | NS_PACK_HELDOUT | NS_PACK_SHUFFLE_ROWS |
                        NS_PACK_WRAP | NS_PACK_HOST_CORPUS | NS_PACK_ORDERED_FREE */
  int32_t pad_id;    /* token written at padded positions */
  uint32_t window_segment; /* G > 0: each stream's windows are read in a shuffled
                              order within segments of G consecutive windows
                              (NeuronSpark-Trainer README, Concepts: the
                              windows of a segment are read in random
                              order); 0: in order; at most
                              NS_MAX_WINDOW_SEGMENT */
  /* Schedule (host, copied): pieces of the horizon with their own rows per
   * update and weights -- an append-only mixture schedule and a batch-size
   * ramp (NeuronSpark-Trainer README, Concepts and Training; Zephon's work
   * source changing the weights during a run).  Piece p covers updates
   * [piece_begin[p], piece_begin[p+1]), the last one up to max_steps.  The
   * quota rule's counts start again at every piece; the windows each stream
   * has given run on.  n_pieces 0: one piece of B rows with source_weight and
   * stream_weight.  With a schedule, B is the largest piece_B (the row stride
   * of the context's tables) and a call may only ask for rows every update it
   * covers has. */
  uint32_t n_pieces;                   /* 0 .. max_steps */
  const uint32_t *piece_begin;         /* [n_pieces], [0] == 0, increasing, < max_steps */
  const uint32_t *piece_B;             /* [n_pieces], 1 .. B */
  const uint32_t *piece_source_weight; /* [n_pieces][n_sources], > 0 */
  const uint32_t *piece_stream_weight; /* [n_pieces][n_streams], > 0 */
  /* Row lengths reported in ns_pack_out.row_len: the row's real positions
   * rounded up to a multiple of len_bucket, at most T (Linnet training docs,
   * Other trainers: packed row lengths are rounded up to a bucket so that few
   * shapes compile); 0 reports the real length. */
  uint32_t len_bucket;
  void *cuda_stream; /* cudaStream_t for init and default for the other calls */
  ns_alloc_fn alloc;
  ns_free_fn free;
  void *alloc_user;
} ns_pack_config;

/* Caller-owned device outputs of ns_pack_step, row-major
 * [n_steps][row_end - row_begin][T]; tokens/pos/doc/mask 16-byte aligned,
 * row_fp 8-byte, row_learned and row_len 4-byte aligned. */
typedef struct {
  int32_t *tokens;
  int32_t *pos;
  int32_t *doc;
  uint8_t *mask;
  uint64_t *row_fp;     /* [n_steps][rows] */
  int32_t *row_learned; /* [n_steps][rows] */
  int32_t *row_len;     /* [n_steps][rows] or NULL: real positions of the row
                           (they come first), rounded up to len_bucket */
} ns_pack_out;

typedef struct {
  uint32_t valid_steps; /* updates [0, valid_steps) can be assembled */
  uint32_t max_steps;
  uint32_t n_streams;
  uint32_t T;
  uint32_t B;
  uint32_t levels;      /* pointer-jumping levels used at init (0: wrap packing) */
  uint64_t order_digest;
  uint64_t n_pieces;    /* pieces built at init: document T-chunks, or whole
                           documents under wrap packing */
  uint64_t table_bytes; /* device bytes the context keeps */
  uint32_t init_launches; /* kernels ns_pack_init launched */
  uint32_t init_passes;   /* 1; 2 when the held-out hash's speculated bound left
                             a stream short of the windows the horizon reads
                             and the context was built again with the full
                             bound (the same tables either way) */
  uint64_t host_bytes;  /* bytes of a host-resident corpus (NS_PACK_HOST_CORPUS)
                           that ns_pack_init read from host memory: offsets,
                           loss starts and the tokens it used (the whole
                           corpus when it had to copy it); 0 otherwise */
  uint64_t hashed_tokens; /* tokens the held-out hash read (every init pass;
                             0 when no source holds documents out) */
  uint64_t hashed_docs;   /* non-empty documents it decided */
  uint64_t hash_ns;       /* device time from the first held-out hash launch to
                             the end of the last one (both rounds, and the fill
                             measurement between them; every init pass), from
                             CUDA events on cfg->cuda_stream; 0 without a hash */
} ns_pack_info_t;

/* Build the context: validate, then on cfg->cuda_stream hash the documents of
 * every source with a held-out rate, shuffle every stream, pack the prefix of
 * each stream that max_steps can reach, number its windows and apportion every
 * update of the horizon.  Defined by: NeuronSpark-Trainer README, Concepts
 * (held out by a hash of the text, the same in every line; documents
 * shuffled; cut at document ends; every source within two samples of its
 * share in every update, strata at theirs; max_epochs 1) and Training (the
 * sample order's digest, ns_pack_info.order_digest, checked on resume).
 * Synchronises the stream twice.  On success
 * *out owns device tables allocated through cfg->alloc; on failure nothing is
 * kept and *out is NULL.  Errors: INVALID_ARG, CUDA, OOM, BAD_INPUT. */
int ns_pack_init(const ns_pack_config *cfg, ns_pack_ctx **out);

/* Assemble rows [row_begin, row_end) of updates [step0, step0 + n_steps) into
 * `out`, asynchronously on cuda_stream (NULL: the context's stream).  One
 * kernel launch.  Defined by: Linnet training docs, Supervised fine-tuning
 * (rows of exactly T positions, padded; completion tokens learned) and Other
 * trainers (a position id of 0 starts a new sequence); "Zephon:
 * deterministic data loading", checkpoint on 16 GPUs and resume on 8/32/64
 * (a batch's bytes do not depend on how its rows are split); per-row
 * fingerprint and learned count in the same pass.  The bytes of every row are the same whatever the row range
 * or the step batching.  Errors: INVALID_ARG (n_steps == 0, empty or out-of-
 * range rows, NULL or misaligned outputs), HORIZON (step0 + n_steps >
 * max_steps), EXHAUSTED (step0 + n_steps > valid_steps), CUDA.  With a
 * schedule, row_end may not exceed the rows of any update of the call. */
int ns_pack_step(ns_pack_ctx *ctx, uint32_t step0, uint32_t n_steps, uint32_t row_begin,
                 uint32_t row_end, const ns_pack_out *out, void *cuda_stream);

/* Fold n_rows row fingerprints (device, in row order) into the batch
 * fingerprint F = fold(F ^ fp_i) and copy it to *batch_fp_host (a hash of
 * every global batch: "Zephon: deterministic data loading", checkpoint on
 * 16 GPUs, resume on 8/32/64); synchronises
 * cuda_stream (NULL: the context's).  Also reports the device error word.
 * Uses one word of the context's memory: calls on one context must not
 * overlap (ns_pack_batch_fp writes to caller memory and has no such limit).
 * Errors: INVALID_ARG (NULL or misaligned pointers, n_rows 0), CUDA, DEVICE,
 * BAD_INPUT. */
int ns_pack_fingerprint(ns_pack_ctx *ctx, const uint64_t *row_fp_dev, uint32_t n_rows,
                        uint64_t *batch_fp_host, void *cuda_stream);

/* Asynchronous variant for n_steps consecutive batches of n_rows rows each:
 * batch_fp_dev[s] = fold of row_fp_dev[s * n_rows .. (s + 1) * n_rows).
 * Errors: INVALID_ARG (NULL or misaligned pointers, n_steps or n_rows 0,
 * n_steps >= 2^31), CUDA. */
int ns_pack_batch_fp(ns_pack_ctx *ctx, const uint64_t *row_fp_dev, uint32_t n_steps,
                     uint32_t n_rows, uint64_t *batch_fp_dev, void *cuda_stream);

/* Learned positions of n_steps consecutive updates of n_rows rows each:
 * learned_dev[s] = sum of row_learned_dev[s * n_rows .. (s + 1) * n_rows)
 * (device int32 in, device int64 out), the count an update's loss is weighed
 * by (Linnet training docs, Supervised fine-tuning).  For a row slice it is
 * the slice's share; the update's count is the sum over its slices.
 * Asynchronous on cuda_stream (NULL: the context's).  Errors: INVALID_ARG
 * (NULL or misaligned pointers, n_steps or n_rows 0, n_steps >= 2^31), CUDA. */
int ns_pack_step_learned(ns_pack_ctx *ctx, const int32_t *row_learned_dev, uint32_t n_steps,
                         uint32_t n_rows, int64_t *learned_dev, void *cuda_stream);

/* Summary of the context (host memory, no synchronisation): the valid
 * horizon (NeuronSpark-Trainer README, Concepts: running out of a source is
 * an error), the order digest (same README, Training), what init read. */
int ns_pack_info(const ns_pack_ctx *ctx, ns_pack_info_t *info);

/* Per stream (host arrays of n_streams; the greedy packing of NeuronSpark-
 * Trainer README, Concepts, cut at document ends): windows packed at init and whether
 * that count is the stream's total (1) or only the prefix the horizon reaches
 * (0, in which case it exceeds every window the horizon asks for). */
int ns_pack_stream_windows(const ns_pack_ctx *ctx, uint64_t *windows, uint8_t *complete);

/* Copy the quota tables (NeuronSpark-Trainer README, Concepts: each source
 * within two samples of its share in every update, strata at theirs) to the
 * host: quota[k][j] windows of stream j in
 * update k (max_steps x n_streams, int32) and cum[k][j] windows before update
 * k ((max_steps + 1) x n_streams, int32).  Either may be NULL.  Synchronises
 * the context's stream.  Errors: INVALID_ARG, CUDA. */
int ns_pack_quota_table(const ns_pack_ctx *ctx, int32_t *quota, int32_t *cum);

/* Synchronise the context's stream and report the device error word (the
 * checks fail fast: "Zephon: deterministic data loading", TorchTitan).
 * Errors: CUDA, DEVICE, BAD_INPUT. */
int ns_pack_check(ns_pack_ctx *ctx);

/* Release every table of the context (NULL is a no-op).  Waits first for
 * the work that may still read them: the device, if ns_pack_step ever ran on
 * a stream other than the context's; else the context's stream, unless the
 * context was built with NS_PACK_ORDERED_FREE (then it does not wait). */
void ns_pack_free(ns_pack_ctx *ctx);

const char *ns_pack_strerror(int code);

/* ---- quota tables without allocating --------------------------------------
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc: a trainer that gives all of the GPU's memory to
 * its own pool at start-up, a process held to a fixed memory budget on a
 * shared GPU, or a loop that cannot afford the device synchronisation that
 * cudaMalloc / cudaFree imply.  It computes the same tables that ns_pack_init
 * builds and ns_pack_quota_table returns -- quota[k][j], the windows of stream
 * j in update k (max_steps x n_streams), and cum[k][j], its windows before
 * update k ((max_steps + 1) x n_streams), both int32 -- into device buffers the
 * caller owns, asynchronously on cuda_stream (NULL: the legacy default
 * stream).  The call only enqueues kernels: the recipe reaches the device in
 * the parameter blocks of small upload kernels (about 7,680 weights each), so
 * no copy from pageable memory waits on the stream, and the caller's arrays
 * may be released as soon as the call returns.
 *
 * Arguments: the recipe's weights on the host (the same meaning and checks as
 * in ns_pack_config: source_weight[n_sources] > 0, stream_source[n_streams]
 * nondecreasing with every source owning 1..NS_MAX_STRATA_PER_SOURCE streams,
 * stream_weight[n_streams] > 0), B >= 1, max_steps >= 1 with max_steps * B <
 * 2^31.  Nothing is allocated: the device copies of the weights and, when
 * there are more than 32 sources or more than 32 strata in a source, a
 * [max_steps][n_sources] int32 table live in one static device array of
 * NS_NOALLOC_SCRATCH_BYTES that every GPU loading this library holds until
 * exit.  A recipe whose scratch does not fit returns NS_ERR_INVALID_ARG, as do
 * out-of-range arguments and quota_dev or cum_dev not 4-byte aligned;
 * NS_ERR_CUDA if a CUDA call fails.  The first call on
 * each device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current) and keeps it: make that first call before any stream
 * capture.  All calls share the array and it keeps the last call's contents;
 * calls whose work overlaps on the GPU (on different streams, or from several
 * threads without ordering) race on it. */
#define NS_NOALLOC_SCRATCH_BYTES (8u << 20)
int ns_pack_quota_noalloc(const uint32_t *source_weight, uint32_t n_sources,
                          const uint32_t *stream_source, const uint32_t *stream_weight,
                          uint32_t n_streams, uint32_t B, uint32_t max_steps,
                          int32_t *quota_dev, int32_t *cum_dev, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* NSPACK_H */
