/*
 * oracle.c -- a plain, sequential CPU statement of deterministic packed
 * assembly: pre-tokenized documents from a weighted mixture of sources become
 * fixed [B, T] global batches that depend only on (seed, step).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg load
 * it.  It shares no code, header, table or helper with the CUDA library, and
 * neither includes nor links the other.  It is written for a reader checking
 * it against the method's definitions by eye: every step walks documents and
 * windows one by one, in the order the definitions state them, with no binary
 * search, jump table, scan or parallelism.
 *
 * Sources of the definitions:
 *  - "NeuronSpark-Trainer" README, Concepts: a held-out split by a hash of a
 *    document's text, 1 % per file (5 % for one source), the same in every
 *    line; documents of a file shuffled; every update holds each source within
 *    two samples of its recipe share; strata of a source at their share; cut
 *    at document ends; max_epochs 1 (running out of a source stops with an error); each
 *    source's validation rows come from the held-out documents of every
 *    stratum (a validation stream packs exactly those); the windows of a
 *    segment are read in a random order.  Training: an append-only mixture
 *    schedule and a batch-size ramp (pieces of the horizon).
 *  - "Zephon: deterministic data loading" (aixai.ru), the section on
 *    checkpointing on 16 GPUs and resuming on 8/32/64: every global batch is
 *    byte-identical (SHA-256) whatever the GPU count.
 *  - Linnet training docs, Supervised fine-tuning: rows of exactly T
 *    positions, padded; only the completion is learned; each step weighs by
 *    its count of learned positions.  Other trainers: a position id of 0
 *    starts a new sequence within a row.  Reinforcement learning / JAX: a
 *    short final step is filled with rows that learn nothing.
 *
 * Where those pages leave a step open, the reading taken is the plainest one:
 *  - the "text" hashed is the document's token ids, position-keyed, with the
 *    SplitMix64 finaliser (Steele, Lea & Flood 2014; Vigna's public-domain
 *    splitmix64.c) as the mixing function; held out iff the hash's high
 *    product with 10000 is below the source's rate in basis points;
 *  - the shuffle is a 4-round balanced Feistel network with cycle walking,
 *    keyed by (seed, stream); positions are permuted first, held-out and empty
 *    documents dropped after;
 *  - a document longer than T is cut into T-chunks from its start, the last
 *    chunk holding the remainder; a piece fits an open window iff the window's
 *    used positions plus its length are at most T;
 *  - the "wrap" variant (Zephon's pipeline example: pack_flat with
 *    algorithm "wrap") concatenates a stream's kept documents and cuts the run
 *    into windows of exactly T tokens, across document ends; a piece is then
 *    a document's run inside one window, and its position ids start at 0;
 *  - quotas are counted in windows (samples), by one largest-remainder rule
 *    applied first to sources, then to each source's strata, with the
 *    cumulative shortfall as the remainder's priority;
 *  - per row, a 64-bit fingerprint: SplitMix64 of the wrapping sum of
 *    SplitMix64 over keyed positions; per batch, a fold of the rows' values.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_INVALID_ARG (-1)
#define OR_ERR_OOM (-3)
#define OR_ERR_EXHAUSTED (-4)
#define OR_ERR_HORIZON (-5)
#define OR_ERR_BAD_INPUT (-6)

#define OR_GOLDEN 0x9E3779B97F4A7C15ull

typedef struct {
  const int32_t *tokens;
  uint64_t n_tokens;
  const int64_t *doc_offsets;   /* [n_docs + 1] */
  const int32_t *loss_start;    /* [n_docs] or NULL: every token learned */
  uint32_t n_docs;
  uint32_t n_sources;
  uint32_t n_streams;
  uint32_t T;
  const uint32_t *stream_doc_begin;  /* [n_streams + 1] */
  const uint32_t *stream_source;     /* [n_streams] */
  const uint32_t *source_weight;     /* [n_sources] */
  const uint32_t *stream_weight;     /* [n_streams] */
  const uint16_t *source_heldout_bp; /* [n_sources] */
  uint64_t seed;
  uint64_t hash_key;
  uint32_t B;
  uint32_t max_steps;
  uint32_t drain;
  int32_t pad_id;
  uint32_t heldout_only; /* 1: pack the held-out documents (the validation stream) */
  uint32_t window_segment; /* G > 0: read each stream's windows in a shuffled order
                              within segments of G windows; 0: in order */
  uint32_t shuffle_rows;   /* 1: rows of an update in a shuffled order */
  /* schedule: pieces [begin_p, begin_{p+1}) of the horizon with their own
     rows per update and weights; 0 pieces: one piece (B and the weights above) */
  uint32_t n_pieces;
  const uint32_t *piece_begin;         /* [n_pieces], [0] == 0, increasing */
  const uint32_t *piece_B;             /* [n_pieces], 1..B */
  const uint32_t *piece_source_weight; /* [n_pieces][n_sources] */
  const uint32_t *piece_stream_weight; /* [n_pieces][n_streams] */
  uint32_t wrap;       /* 1: windows are consecutive T-token cuts of the stream's
                          kept tokens, across document ends */
  uint32_t len_bucket; /* row length reported as the real length rounded up to a
                          multiple of this (0: the real length) */
} or_config;

typedef struct {
  uint32_t doc; /* global document index */
  uint32_t off; /* offset of the piece inside its document (a multiple of T
                   under greedy packing; anywhere under wrap packing) */
  uint32_t len; /* 1..T */
} or_piece;

typedef struct {
  or_piece *pieces;
  uint64_t n_pieces;
  uint64_t *win_first; /* [n_windows + 1]: window r is pieces [first[r], first[r+1]) */
  uint64_t n_windows;
} or_stream;

typedef struct {
  or_config cfg;
  uint64_t *doc_hash;  /* [n_docs] (0 for documents no held-out rate applies to) */
  uint8_t *heldout;    /* [n_docs] */
  or_stream *streams;  /* [n_streams] */
  int64_t *quota;      /* [max_steps][n_streams]: windows of stream j in step k */
  int64_t *cum;        /* [max_steps + 1][n_streams]: windows before step k */
  int64_t *src_quota;  /* [max_steps][n_sources] */
  uint32_t valid_steps;
  uint64_t digest;
} or_ctx;

/* ---- SplitMix64 finaliser, as a pure function of x --------------------- */
uint64_t or_splitmix64(uint64_t x) {
  uint64_t z = x + OR_GOLDEN;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* ---- held-out split by a hash of the document's text -------------------
 * acc = sum over i < L of splitmix64((i << 32) | (u32)tok_i)   (mod 2^64)
 * h   = splitmix64(acc ^ splitmix64(hash_key + L))                       */
uint64_t or_doc_hash(const int32_t *tok, uint64_t len, uint64_t hash_key) {
  uint64_t acc = 0;
  for (uint64_t i = 0; i < len; i++)
    acc += or_splitmix64((i << 32) | (uint64_t)(uint32_t)tok[i]);
  return or_splitmix64(acc ^ or_splitmix64(hash_key + len));
}

/* held out iff floor(h * 10000 / 2^64) < bp */
int or_is_heldout(uint64_t h, uint32_t bp) {
  unsigned __int128 prod = (unsigned __int128)h * 10000u;
  return (uint64_t)(prod >> 64) < (uint64_t)bp;
}

/* ---- the shuffle: a keyed Feistel permutation of [0, N) ----------------- */
uint32_t or_feistel_bits(uint64_t n) {
  uint32_t b = 0;
  while (b < 64 && (1ull << b) < n) b++;
  if (b < 2) b = 2;
  if (b & 1) b++;
  return b;
}

uint64_t or_feistel_round_key(uint64_t seed, uint32_t stream, uint32_t round) {
  return or_splitmix64(or_splitmix64(seed) ^
                       or_splitmix64(((uint64_t)stream << 8) | round));
}

/* one pass of the 4-round network over a domain of 2 * half bits */
uint64_t or_feistel_encrypt(const uint64_t key[4], uint32_t half, uint64_t x) {
  uint64_t mask = (half >= 64) ? ~0ull : ((1ull << half) - 1);
  uint64_t L = x >> half, R = x & mask;
  for (int r = 0; r < 4; r++) {
    uint64_t F = or_splitmix64(key[r] ^ R) & mask;
    uint64_t nl = R, nr = L ^ F;
    L = nl;
    R = nr;
  }
  return (L << half) | R;
}

/* position p of stream j -> index of the document it reads (cycle walking) */
uint64_t or_feistel_pi(uint64_t seed, uint32_t stream, uint64_t n, uint64_t p) {
  uint64_t key[4];
  for (uint32_t r = 0; r < 4; r++) key[r] = or_feistel_round_key(seed, stream, r);
  uint32_t half = or_feistel_bits(n) / 2;
  uint64_t y = or_feistel_encrypt(key, half, p);
  while (y >= n) y = or_feistel_encrypt(key, half, y);
  return y;
}

/* ---- the order in which windows and rows are read ----------------------
 * The trainer reads the windows of a segment of each source in random order
 * (NeuronSpark-Trainer README, Concepts).  With a window segment of G > 0 the
 * windows of stream j are grouped in segments of G consecutive windows (the
 * last one shorter); rank r of segment s = r / G reads window
 * sG + sigma_{j,s}(r - sG), sigma the same keyed Feistel network as the
 * document shuffle over the segment's length, keyed by (seed + 1, j, s).
 * With row shuffling, slot i of update k holds the row that would otherwise
 * be row rho_k(i), rho_k the same network over [0, B) keyed by (seed + 2, k). */
uint64_t or_window_round_key(uint64_t seed, uint32_t stream, uint64_t segment, uint32_t round) {
  return or_splitmix64(or_splitmix64(seed + 1) ^
                       or_splitmix64(((uint64_t)stream << 40) | (segment << 8) | round));
}

uint64_t or_row_round_key(uint64_t seed, uint32_t step, uint32_t round) {
  return or_splitmix64(or_splitmix64(seed + 2) ^ or_splitmix64(((uint64_t)step << 8) | round));
}

static uint64_t walk(const uint64_t key[4], uint64_t n, uint64_t p) {
  uint32_t half = or_feistel_bits(n) / 2;
  uint64_t y = or_feistel_encrypt(key, half, p);
  while (y >= n) y = or_feistel_encrypt(key, half, y);
  return y;
}

/* window read by rank r of a stream with W windows */
uint64_t or_window_of_rank(uint64_t seed, uint32_t stream, uint32_t G, uint64_t W, uint64_t r) {
  if (G == 0) return r;
  uint64_t s = r / G, b = s * G;
  uint64_t n = (W - b < G) ? (W - b) : G;
  uint64_t key[4];
  for (uint32_t q = 0; q < 4; q++) key[q] = or_window_round_key(seed, stream, s, q);
  return b + walk(key, n, r - b);
}

/* row held by slot i of update k */
uint32_t or_row_of_slot(uint64_t seed, uint32_t step, uint32_t B, uint32_t i) {
  uint64_t key[4];
  for (uint32_t q = 0; q < 4; q++) key[q] = or_row_round_key(seed, step, q);
  return (uint32_t)walk(key, B, i);
}

/* ---- per-update apportionment: one level of the quota rule -------------
 * A parent hands out n units at this update (N of them counting every update
 * so far, this one included) among children with weights v (sum V) that hold
 * C units before this update:
 *   base_c  = floor(n * v_c / V),  R = n - sum base_c,
 *   delta_c = N * v_c - V * (C_c + base_c)          (exact),
 *   the R children with the largest delta get one more (ties: lower index). */
int or_apportion(uint32_t n_children, const uint64_t *v, const int64_t *C,
                 int64_t n, int64_t N, int64_t *out) {
  if (n_children == 0 || n < 0) return OR_ERR_INVALID_ARG;
  __int128 V = 0;
  for (uint32_t c = 0; c < n_children; c++) V += (__int128)v[c];
  if (V <= 0) return OR_ERR_INVALID_ARG;
  int64_t given = 0;
  for (uint32_t c = 0; c < n_children; c++) {
    out[c] = (int64_t)(((__int128)n * (__int128)v[c]) / V);
    given += out[c];
  }
  int64_t R = n - given;
  __int128 *delta = (__int128 *)malloc(sizeof(__int128) * n_children);
  uint8_t *chosen = (uint8_t *)calloc(n_children, 1);
  if (!delta || !chosen) {
    free(delta);
    free(chosen);
    return OR_ERR_OOM;
  }
  for (uint32_t c = 0; c < n_children; c++)
    delta[c] = (__int128)N * (__int128)v[c] - V * (__int128)(C[c] + out[c]);
  for (int64_t pick = 0; pick < R; pick++) {
    int64_t best = -1;
    for (uint32_t c = 0; c < n_children; c++) {
      if (chosen[c]) continue;
      if (best < 0 || delta[c] > delta[best]) best = c;
    }
    chosen[best] = 1;
    out[best] += 1;
  }
  free(delta);
  free(chosen);
  return OR_OK;
}

/* ---- the schedule ------------------------------------------------------- */
static uint32_t piece_of(const or_config *c, uint32_t k) {
  uint32_t p = 0;
  for (uint32_t q = 0; q < c->n_pieces; q++)
    if (c->piece_begin[q] <= k) p = q;
  return p;
}
static uint32_t piece_begin(const or_config *c, uint32_t p) {
  return c->n_pieces ? c->piece_begin[p] : 0;
}
static uint32_t rows_of_piece(const or_config *c, uint32_t p) {
  return c->n_pieces ? c->piece_B[p] : c->B;
}
static uint64_t source_w(const or_config *c, uint32_t p, uint32_t s) {
  return c->n_pieces ? c->piece_source_weight[(size_t)p * c->n_sources + s] : c->source_weight[s];
}
static uint64_t stream_w(const or_config *c, uint32_t p, uint32_t j) {
  return c->n_pieces ? c->piece_stream_weight[(size_t)p * c->n_streams + j] : c->stream_weight[j];
}
/* rows of update k */
uint32_t or_rows_of_step(const or_config *c, uint32_t k) { return rows_of_piece(c, piece_of(c, k)); }

/* ---- checks of the recipe and of the corpus ----------------------------- */
static int check_config(const or_config *c) {
  if (!c || !c->tokens || !c->doc_offsets || !c->stream_doc_begin || !c->stream_source ||
      !c->source_weight || !c->stream_weight || !c->source_heldout_bp)
    return OR_ERR_INVALID_ARG;
  if (c->T == 0 || c->T > (1u << 24)) return OR_ERR_INVALID_ARG;
  if (c->B == 0 || c->max_steps == 0) return OR_ERR_INVALID_ARG;
  if ((uint64_t)c->max_steps * c->B >= (1ull << 31)) return OR_ERR_INVALID_ARG;
  if (c->n_sources == 0 || c->n_streams == 0) return OR_ERR_INVALID_ARG;
  if (c->n_docs >= (1u << 31)) return OR_ERR_INVALID_ARG;
  for (uint32_t s = 0; s < c->n_sources; s++) {
    if (c->source_weight[s] == 0 || c->source_heldout_bp[s] > 10000) return OR_ERR_INVALID_ARG;
  }
  for (uint32_t j = 0; j < c->n_streams; j++) {
    if (c->stream_weight[j] == 0 || c->stream_source[j] >= c->n_sources) return OR_ERR_INVALID_ARG;
    if (j > 0 && c->stream_source[j] < c->stream_source[j - 1]) return OR_ERR_INVALID_ARG;
    if (c->stream_doc_begin[j + 1] < c->stream_doc_begin[j]) return OR_ERR_INVALID_ARG;
  }
  if (c->stream_doc_begin[c->n_streams] > c->n_docs) return OR_ERR_INVALID_ARG;
  /* every source owns at least one stream */
  for (uint32_t s = 0; s < c->n_sources; s++) {
    int found = 0;
    for (uint32_t j = 0; j < c->n_streams; j++) found |= (c->stream_source[j] == s);
    if (!found) return OR_ERR_INVALID_ARG;
  }
  /* the schedule: pieces start at 0, in increasing order, inside the horizon */
  if (c->n_pieces) {
    if (!c->piece_begin || !c->piece_B || !c->piece_source_weight || !c->piece_stream_weight)
      return OR_ERR_INVALID_ARG;
    if (c->n_pieces > c->max_steps || c->piece_begin[0] != 0) return OR_ERR_INVALID_ARG;
    for (uint32_t p = 0; p < c->n_pieces; p++) {
      if (p > 0 && c->piece_begin[p] <= c->piece_begin[p - 1]) return OR_ERR_INVALID_ARG;
      if (c->piece_begin[p] >= c->max_steps) return OR_ERR_INVALID_ARG;
      if (c->piece_B[p] == 0 || c->piece_B[p] > c->B) return OR_ERR_INVALID_ARG;
      for (uint32_t s = 0; s < c->n_sources; s++)
        if (c->piece_source_weight[(size_t)p * c->n_sources + s] == 0) return OR_ERR_INVALID_ARG;
      for (uint32_t j = 0; j < c->n_streams; j++)
        if (c->piece_stream_weight[(size_t)p * c->n_streams + j] == 0) return OR_ERR_INVALID_ARG;
    }
  }
  /* the corpus: offsets start in range, never decrease, end inside the tokens */
  if (c->doc_offsets[0] < 0) return OR_ERR_BAD_INPUT;
  for (uint32_t d = 0; d < c->n_docs; d++) {
    int64_t len = c->doc_offsets[d + 1] - c->doc_offsets[d];
    if (len < 0 || len > 0x7FFFFFFF) return OR_ERR_BAD_INPUT;
  }
  if ((uint64_t)c->doc_offsets[c->n_docs] > c->n_tokens) return OR_ERR_BAD_INPUT;
  return OR_OK;
}

static uint64_t doc_len(const or_config *c, uint32_t d) {
  return (uint64_t)(c->doc_offsets[d + 1] - c->doc_offsets[d]);
}

/* ---- greedy packing of one stream, walked document by document ---------- */
static int pack_stream(or_ctx *x, uint32_t j) {
  const or_config *c = &x->cfg;
  or_stream *st = &x->streams[j];
  uint32_t d0 = c->stream_doc_begin[j];
  uint64_t n = (uint64_t)c->stream_doc_begin[j + 1] - d0;
  uint64_t cap_p = 16, cap_w = 16;
  st->pieces = (or_piece *)malloc(sizeof(or_piece) * cap_p);
  st->win_first = (uint64_t *)malloc(sizeof(uint64_t) * cap_w);
  if (!st->pieces || !st->win_first) return OR_ERR_OOM;
  st->n_pieces = 0;
  st->n_windows = 0;
  uint64_t key[4];
  for (uint32_t r = 0; r < 4; r++) key[r] = or_feistel_round_key(c->seed, j, r);
  uint32_t half = or_feistel_bits(n) / 2;
  uint64_t used = 0; /* positions used in the open window (0: none open) */
  for (uint64_t p = 0; p < n; p++) {
    uint64_t y = or_feistel_encrypt(key, half, p);
    while (y >= n) y = or_feistel_encrypt(key, half, y);
    uint32_t d = d0 + (uint32_t)y;
    uint64_t L = doc_len(c, d);
    /* the training stream keeps what is not held out; the validation stream
       keeps exactly what is */
    if (L == 0 || x->heldout[d] != (c->heldout_only ? 1 : 0)) continue;
    for (uint64_t off = 0; off < L;) {
      uint64_t len;
      if (c->wrap) {
        /* concatenate and cut: the piece runs to the document's end or to
           the window's, whichever comes first */
        len = L - off;
        if (len > c->T - used) len = c->T - used;
      } else {
        /* greedy, cut at document ends: T-chunks from the document's start;
           a piece that does not fit closes the window (the rest is padding) */
        len = (L - off < c->T) ? (L - off) : c->T;
        if (used + len > c->T) used = 0;
      }
      if (used == 0) {                  /* open a new window at this piece */
        if (st->n_windows + 1 >= cap_w) {
          cap_w *= 2;
          uint64_t *w = (uint64_t *)realloc(st->win_first, sizeof(uint64_t) * cap_w);
          if (!w) return OR_ERR_OOM;
          st->win_first = w;
        }
        st->win_first[st->n_windows++] = st->n_pieces;
      }
      if (st->n_pieces == cap_p) {
        cap_p *= 2;
        or_piece *q = (or_piece *)realloc(st->pieces, sizeof(or_piece) * cap_p);
        if (!q) return OR_ERR_OOM;
        st->pieces = q;
      }
      st->pieces[st->n_pieces].doc = d;
      st->pieces[st->n_pieces].off = (uint32_t)off;
      st->pieces[st->n_pieces].len = (uint32_t)len;
      st->n_pieces++;
      used += len;
      off += len;
      if (c->wrap && used == c->T) used = 0; /* a full window closes */
    }
  }
  st->win_first[st->n_windows] = st->n_pieces;
  return OR_OK;
}

/* ---- quotas for every update: sources first, then strata of each source --
 * A schedule splits the horizon into pieces with their own weights and rows
 * per update (an append-only mixture schedule, a batch-size ramp): the rule's
 * counts (N, and every child's C) start again from 0 at each piece, while the
 * windows each stream has given (cum) run on across pieces.  Without a
 * schedule the whole horizon is one piece. */
static int build_quotas(or_ctx *x) {
  const or_config *c = &x->cfg;
  uint32_t S = c->n_sources, J = c->n_streams, K = c->max_steps;
  x->quota = (int64_t *)calloc((size_t)K * J, sizeof(int64_t));
  x->cum = (int64_t *)calloc((size_t)(K + 1) * J, sizeof(int64_t));
  x->src_quota = (int64_t *)calloc((size_t)K * S, sizeof(int64_t));
  uint64_t *vs = (uint64_t *)malloc(sizeof(uint64_t) * S);
  int64_t *Cs = (int64_t *)calloc(S, sizeof(int64_t));      /* per piece */
  int64_t *Cj = (int64_t *)calloc(J, sizeof(int64_t));      /* per piece */
  uint64_t *vt = (uint64_t *)malloc(sizeof(uint64_t) * J);
  int64_t *Ct = (int64_t *)malloc(sizeof(int64_t) * J);
  int64_t *at = (int64_t *)malloc(sizeof(int64_t) * J);
  int rc = OR_OK;
  if (!x->quota || !x->cum || !x->src_quota || !vs || !Cs || !Cj || !vt || !Ct || !at) {
    rc = OR_ERR_OOM;
    goto done;
  }
  for (uint32_t k = 0; k < K; k++) {
    uint32_t p = piece_of(c, k);
    uint32_t k0 = piece_begin(c, p);
    int64_t Bk = rows_of_piece(c, p);
    if (k == k0) {
      memset(Cs, 0, sizeof(int64_t) * S);
      memset(Cj, 0, sizeof(int64_t) * J);
    }
    for (uint32_t s = 0; s < S; s++) vs[s] = source_w(c, p, s);
    int64_t *as = x->src_quota + (size_t)k * S;
    rc = or_apportion(S, vs, Cs, Bk, (int64_t)(k - k0 + 1) * Bk, as);
    if (rc) goto done;
    for (uint32_t s = 0; s < S; s++) {
      uint32_t n_st = 0, j0 = 0;
      for (uint32_t j = 0; j < J; j++) {
        if (c->stream_source[j] != s) continue;
        if (n_st == 0) j0 = j;
        vt[n_st] = stream_w(c, p, j);
        Ct[n_st] = Cj[j];
        n_st++;
      }
      rc = or_apportion(n_st, vt, Ct, as[s], Cs[s] + as[s], at);
      if (rc) goto done;
      for (uint32_t t = 0; t < n_st; t++) {
        x->quota[(size_t)k * J + j0 + t] = at[t];
        Cj[j0 + t] += at[t];
      }
      Cs[s] += as[s];
    }
    for (uint32_t j = 0; j < J; j++)
      x->cum[(size_t)(k + 1) * J + j] = x->cum[(size_t)k * J + j] + x->quota[(size_t)k * J + j];
  }
done:
  free(vs);
  free(Cs);
  free(Cj);
  free(vt);
  free(Ct);
  free(at);
  return rc;
}

/* ---- the order digest: what a resumed run compares before it continues --- */
typedef struct {
  uint64_t sum;
  uint64_t count;
} digest_acc;

static void digest_add(digest_acc *a, uint64_t item) {
  a->sum += or_splitmix64(item ^ or_splitmix64(a->count));
  a->count++;
}

static uint64_t build_digest(const or_ctx *x) {
  const or_config *c = &x->cfg;
  uint32_t J = c->n_streams;
  digest_acc a = {0, 0};
  digest_add(&a, c->T);
  digest_add(&a, c->B);
  digest_add(&a, c->max_steps);
  digest_add(&a, x->valid_steps);
  digest_add(&a, (c->drain ? 1u : 0u) | (c->heldout_only ? 2u : 0u) | (c->shuffle_rows ? 4u : 0u) |
                    (c->wrap ? 8u : 0u));
  digest_add(&a, (uint64_t)(uint32_t)c->pad_id);
  digest_add(&a, c->seed);
  digest_add(&a, c->hash_key);
  digest_add(&a, c->n_sources);
  digest_add(&a, c->n_streams);
  digest_add(&a, c->window_segment);
  digest_add(&a, c->len_bucket);
  for (uint32_t s = 0; s < c->n_sources; s++) {
    digest_add(&a, c->source_weight[s]);
    digest_add(&a, c->source_heldout_bp[s]);
  }
  for (uint32_t j = 0; j < J; j++) {
    digest_add(&a, c->stream_doc_begin[j]);
    digest_add(&a, c->stream_doc_begin[j + 1]);
    digest_add(&a, c->stream_source[j]);
    digest_add(&a, c->stream_weight[j]);
  }
  if (c->n_pieces) {
    digest_add(&a, c->n_pieces);
    for (uint32_t p = 0; p < c->n_pieces; p++) {
      digest_add(&a, c->piece_begin[p]);
      digest_add(&a, c->piece_B[p]);
      for (uint32_t s = 0; s < c->n_sources; s++) digest_add(&a, source_w(c, p, s));
      for (uint32_t j = 0; j < J; j++) digest_add(&a, stream_w(c, p, j));
    }
  }
  for (uint32_t k = 0; k < x->valid_steps; k++)
    for (uint32_t j = 0; j < J; j++) digest_add(&a, (uint64_t)x->quota[(size_t)k * J + j]);
  for (uint32_t j = 0; j < J; j++) {
    const or_stream *st = &x->streams[j];
    uint64_t used = (uint64_t)x->cum[(size_t)x->valid_steps * J + j];
    if (used > st->n_windows) used = st->n_windows;
    for (uint64_t r = 0; r < used; r++) {
      uint64_t w = or_window_of_rank(c->seed, j, c->window_segment, st->n_windows, r);
      const or_piece *p = &st->pieces[st->win_first[w]];
      digest_add(&a, ((uint64_t)p->doc << 32) | (uint64_t)p->off);
    }
  }
  return or_splitmix64(a.sum ^ a.count);
}

/* ---- build: hash, shuffle, pack, apportion ------------------------------ */
void or_free(or_ctx *x) {
  if (!x) return;
  if (x->streams) {
    for (uint32_t j = 0; j < x->cfg.n_streams; j++) {
      free(x->streams[j].pieces);
      free(x->streams[j].win_first);
    }
  }
  free(x->streams);
  free(x->doc_hash);
  free(x->heldout);
  free(x->quota);
  free(x->cum);
  free(x->src_quota);
  free(x);
}

int or_build(const or_config *cfg, or_ctx **out) {
  if (!out) return OR_ERR_INVALID_ARG;
  *out = NULL;
  int rc = check_config(cfg);
  if (rc) return rc;
  or_ctx *x = (or_ctx *)calloc(1, sizeof(or_ctx));
  if (!x) return OR_ERR_OOM;
  x->cfg = *cfg;
  const or_config *c = &x->cfg;
  uint32_t J = c->n_streams;
  x->doc_hash = (uint64_t *)calloc(c->n_docs ? c->n_docs : 1, sizeof(uint64_t));
  x->heldout = (uint8_t *)calloc(c->n_docs ? c->n_docs : 1, 1);
  x->streams = (or_stream *)calloc(J, sizeof(or_stream));
  if (!x->doc_hash || !x->heldout || !x->streams) {
    or_free(x);
    return OR_ERR_OOM;
  }
  /* 1. held-out flags, for every document of a stream whose source holds out */
  for (uint32_t j = 0; j < J; j++) {
    uint32_t bp = c->source_heldout_bp[c->stream_source[j]];
    if (bp == 0) continue;
    for (uint32_t d = c->stream_doc_begin[j]; d < c->stream_doc_begin[j + 1]; d++) {
      uint64_t h = or_doc_hash(c->tokens + c->doc_offsets[d], doc_len(c, d), c->hash_key);
      x->doc_hash[d] = h;
      x->heldout[d] = (uint8_t)or_is_heldout(h, bp);
    }
  }
  /* 2-3. shuffle and pack every stream */
  for (uint32_t j = 0; j < J; j++) {
    rc = pack_stream(x, j);
    if (rc) {
      or_free(x);
      return rc;
    }
  }
  /* 4. quotas for every update of the horizon */
  rc = build_quotas(x);
  if (rc) {
    or_free(x);
    return rc;
  }
  /* 5. the first update that asks a stream for a window it does not have */
  x->valid_steps = c->max_steps;
  for (uint32_t k = 0; k < c->max_steps; k++) {
    int short_of_windows = 0;
    for (uint32_t j = 0; j < J; j++)
      if ((uint64_t)x->cum[(size_t)(k + 1) * J + j] > x->streams[j].n_windows) short_of_windows = 1;
    if (short_of_windows) {
      x->valid_steps = c->drain ? k + 1 : k;
      break;
    }
  }
  x->digest = build_digest(x);
  *out = x;
  return OR_OK;
}

/* ---- the fingerprint of one row of T positions --------------------------
 * key_t = a_t ^ ((b_t | t << 40) * golden), a_t = (u32 tok << 32) | u32 doc,
 * b_t = (mask << 32) | u32 pos; fp = splitmix64(sum of splitmix64(key_t)). */
uint64_t or_row_fp(const int32_t *tok, const int32_t *pos, const int32_t *doc,
                   const uint8_t *mask, uint32_t T) {
  uint64_t acc = 0;
  for (uint32_t t = 0; t < T; t++) {
    uint64_t a = ((uint64_t)(uint32_t)tok[t] << 32) | (uint64_t)(uint32_t)doc[t];
    uint64_t b = ((uint64_t)mask[t] << 32) | (uint64_t)(uint32_t)pos[t];
    uint64_t key = a ^ ((b | ((uint64_t)t << 40)) * OR_GOLDEN);
    acc += or_splitmix64(key);
  }
  return or_splitmix64(acc);
}

/* ---- assembly of rows [row0, row1) of update `step` ----------------------
 * Each row also reports its length: its real positions (the window's tokens,
 * which come first), rounded up to a multiple of len_bucket when that is set
 * (Linnet training docs, Other trainers: packed row lengths are rounded up to
 * a bucket so that few shapes compile).
 * Rows are ordered by (source, stratum, rank), unless shuffled; a rank reads
 * its window through the window order above.  A window's pieces are copied
 * in order; pos is the offset inside the piece (0 starts a new sequence);
 * doc is the global document index; mask is 1 iff the token's offset in its
 * document is at or past loss_start; the tail is pad_id / 0 / -1 / 0.  A row
 * whose window lies past the end of its stream (only in the final, drained
 * update) is all padding.  Outputs are [row1 - row0][T]. */
int or_rows(const or_ctx *x, uint32_t step, uint32_t row0, uint32_t row1, int32_t *tok,
            int32_t *pos, int32_t *doc, uint8_t *mask, uint64_t *row_fp,
            int32_t *row_learned, int32_t *row_len) {
  const or_config *c = &x->cfg;
  uint32_t J = c->n_streams, T = c->T;
  if (step >= c->max_steps) return OR_ERR_HORIZON;
  const uint32_t Bk = or_rows_of_step(c, step);
  if (row0 >= row1 || row1 > Bk) return OR_ERR_INVALID_ARG;
  if (step >= x->valid_steps) return OR_ERR_EXHAUSTED;
  for (uint32_t i = row0; i < row1; i++) {
    size_t o = (size_t)(i - row0) * T;
    /* which stream and which of its windows this row takes */
    uint32_t row = c->shuffle_rows ? or_row_of_slot(c->seed, step, Bk, i) : i;
    uint32_t base = 0, j = 0;
    while (j < J && row >= base + (uint32_t)x->quota[(size_t)step * J + j]) {
      base += (uint32_t)x->quota[(size_t)step * J + j];
      j++;
    }
    uint64_t r = (uint64_t)x->cum[(size_t)step * J + j] + (row - base);
    const or_stream *st = &x->streams[j];
    uint32_t t = 0;
    if (r < st->n_windows) {
      uint64_t w = or_window_of_rank(c->seed, j, c->window_segment, st->n_windows, r);
      for (uint64_t q = st->win_first[w]; q < st->win_first[w + 1]; q++) {
        const or_piece *p = &st->pieces[q];
        const int32_t *src = c->tokens + c->doc_offsets[p->doc] + p->off;
        int64_t ls = c->loss_start ? c->loss_start[p->doc] : 0;
        for (uint32_t e = 0; e < p->len; e++, t++) {
          tok[o + t] = src[e];
          pos[o + t] = (int32_t)e;
          doc[o + t] = (int32_t)p->doc;
          mask[o + t] = ((int64_t)p->off + e >= ls) ? 1 : 0;
        }
      }
    }
    /* the row's length: its real positions, rounded up to the bucket */
    uint32_t len = t;
    if (c->len_bucket) {
      len = (t + c->len_bucket - 1) / c->len_bucket * c->len_bucket;
      if (len > T) len = T;
    }
    row_len[i - row0] = (int32_t)len;
    for (; t < T; t++) {
      tok[o + t] = c->pad_id;
      pos[o + t] = 0;
      doc[o + t] = -1;
      mask[o + t] = 0;
    }
    row_fp[i - row0] = or_row_fp(tok + o, pos + o, doc + o, mask + o, T);
    int32_t learned = 0;
    for (t = 0; t < T; t++) learned += mask[o + t];
    row_learned[i - row0] = learned;
  }
  return OR_OK;
}

/* fold of the row fingerprints, in row order */
uint64_t or_batch_fp(const uint64_t *row_fp, uint32_t n_rows) {
  uint64_t F = 0;
  for (uint32_t i = 0; i < n_rows; i++) F = or_splitmix64(F ^ row_fp[i]);
  return F;
}

/* ---- read-outs for the tests ------------------------------------------- */
uint32_t or_valid_steps(const or_ctx *x) { return x->valid_steps; }
uint64_t or_digest(const or_ctx *x) { return x->digest; }
uint64_t or_stream_windows(const or_ctx *x, uint32_t j) { return x->streams[j].n_windows; }
uint64_t or_stream_pieces(const or_ctx *x, uint32_t j) { return x->streams[j].n_pieces; }

void or_get_pieces(const or_ctx *x, uint32_t j, uint32_t *doc, uint32_t *off, uint32_t *len) {
  const or_stream *st = &x->streams[j];
  for (uint64_t q = 0; q < st->n_pieces; q++) {
    doc[q] = st->pieces[q].doc;
    off[q] = st->pieces[q].off;
    len[q] = st->pieces[q].len;
  }
}

void or_get_window_first(const or_ctx *x, uint32_t j, uint64_t *first) {
  memcpy(first, x->streams[j].win_first, sizeof(uint64_t) * (x->streams[j].n_windows + 1));
}

void or_get_heldout(const or_ctx *x, uint8_t *out, uint64_t *hash) {
  memcpy(out, x->heldout, x->cfg.n_docs);
  if (hash) memcpy(hash, x->doc_hash, sizeof(uint64_t) * x->cfg.n_docs);
}

void or_get_quota(const or_ctx *x, int64_t *quota, int64_t *cum, int64_t *src_quota) {
  size_t K = x->cfg.max_steps, J = x->cfg.n_streams, S = x->cfg.n_sources;
  if (quota) memcpy(quota, x->quota, sizeof(int64_t) * K * J);
  if (cum) memcpy(cum, x->cum, sizeof(int64_t) * (K + 1) * J);
  if (src_quota) memcpy(src_quota, x->src_quota, sizeof(int64_t) * K * S);
}
