"""A second, independent statement of deterministic packed assembly in plain
Python, for small corpora only.

Test infrastructure: it is written from the method's definitions (the
readings the design notes list), not from the C oracle, and shares nothing
with it or with the CUDA library; tests compare the two oracles byte for byte
on shrunk corpora, so a slip in either one shows up as a disagreement.

Sources of the definitions: NeuronSpark-Trainer README, Concepts (held-out
split by a hash of the text; shuffled documents; each source within two
samples of its share per update, strata at theirs; cut at document ends; the
windows of a segment in random order; validation rows from the held-out
documents) and Training (append-only schedules, batch-size ramps);
"Zephon: deterministic data loading" (the batch hash; the wrap packing of
its pipeline example); Linnet training docs, Supervised fine-tuning and
Other trainers (rows of exactly T positions, completion-only loss, position
ids restarting at 0, packed lengths rounded up to a bucket).
"""
from __future__ import annotations

from dataclasses import dataclass, field

M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15


def mix(x: int) -> int:
    """SplitMix64's output function (Steele, Lea & Flood 2014)."""
    z = (x + GOLDEN) & M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def u32(v: int) -> int:
    return v & 0xFFFFFFFF


# ---- held-out split -------------------------------------------------------
def text_hash(tokens, hash_key: int) -> int:
    s = 0
    for i, t in enumerate(tokens):
        s = (s + mix((i << 32) | u32(int(t)))) & M64
    return mix(s ^ mix((hash_key + len(tokens)) & M64))


def held_out(h: int, bp: int) -> bool:
    return (h * 10000) >> 64 < bp


# ---- keyed permutations ---------------------------------------------------
class Permutation:
    """A 4-round balanced Feistel network on an even number of bits, walked
    until it lands inside [0, n)."""

    def __init__(self, n: int, keys):
        bits = max(2, (n - 1).bit_length() if n > 1 else 0)
        bits += bits % 2
        self.n, self.h = n, bits // 2
        self.mask = (1 << self.h) - 1
        self.keys = keys

    def _once(self, x: int) -> int:
        left, right = x >> self.h, x & self.mask
        for k in self.keys:
            left, right = right, left ^ (mix(k ^ right) & self.mask)
        return (left << self.h) | right

    def __call__(self, p: int) -> int:
        y = self._once(p)
        while y >= self.n:
            y = self._once(y)
        return y


def doc_keys(seed, j):
    return [mix(mix(seed) ^ mix((j << 8) | r)) for r in range(4)]


def segment_keys(seed, j, s):
    return [mix(mix((seed + 1) & M64) ^ mix((j << 40) | (s << 8) | r)) for r in range(4)]


def row_keys(seed, k):
    return [mix(mix((seed + 2) & M64) ^ mix((k << 8) | r)) for r in range(4)]


# ---- packing --------------------------------------------------------------
@dataclass
class Piece:
    doc: int
    off: int     # first token's offset inside the document
    length: int


def pack_greedy(docs, lengths, T):
    """Windows of pieces: documents cut into T-chunks from their start; a
    piece that does not fit the open window closes it."""
    windows, cur, used = [], [], 0
    for d in docs:
        for off in range(0, lengths[d], T):
            n = min(T, lengths[d] - off)
            if used + n > T:
                windows.append(cur)
                cur, used = [], 0
            cur.append(Piece(d, off, n))
            used += n
    if cur:
        windows.append(cur)
    return windows


def pack_wrap(docs, lengths, T):
    """Windows of exactly T tokens cut from the documents laid end to end."""
    windows, cur, used = [], [], 0
    for d in docs:
        off = 0
        while off < lengths[d]:
            n = min(lengths[d] - off, T - used)
            cur.append(Piece(d, off, n))
            used += n
            off += n
            if used == T:
                windows.append(cur)
                cur, used = [], 0
    if cur:
        windows.append(cur)
    return windows


# ---- apportionment --------------------------------------------------------
def apportion(n: int, N: int, weights, before):
    """n units now (N counting this update and the earlier ones of the
    piece) among children holding `before` units: each gets floor(n v / V),
    the remainder goes to the largest cumulative shortfalls N v - V (C +
    base), ties to the lower index."""
    V = sum(weights)
    base = [n * v // V for v in weights]
    short = [N * v - V * (c + b) for v, c, b in zip(weights, before, base)]
    order = sorted(range(len(weights)), key=lambda c: (-short[c], c))
    for c in order[:n - sum(base)]:
        base[c] += 1
    return base


@dataclass
class Twin:
    corpus: object
    seed: int
    hash_key: int
    T: int
    B: int
    K: int
    drain: bool
    pad_id: int
    heldout_only: bool = False
    window_segment: int = 0
    shuffle_rows: bool = False
    schedule: list | None = None
    wrap: bool = False
    len_bucket: int = 0
    windows: list = field(default_factory=list)
    quota: list = field(default_factory=list)
    cum: list = field(default_factory=list)
    valid_steps: int = 0

    # -- schedule pieces -----------------------------------------------------
    def _pieces(self):
        c = self.corpus
        if not self.schedule:
            return [dict(begin=0, B=self.B, source_weight=list(c.source_weight),
                         stream_weight=list(c.stream_weight))]
        return self.schedule

    def rows_of(self, k):
        return [p for p in self._pieces() if p["begin"] <= k][-1]["B"]

    def build(self):
        c = self.corpus
        offs = [int(x) for x in c.doc_offsets]
        toks = c.tokens
        lengths = [offs[d + 1] - offs[d] for d in range(len(offs) - 1)]
        sdb = [int(x) for x in c.stream_doc_begin]
        ssrc = [int(x) for x in c.stream_source]
        J, S = len(ssrc), len(c.source_weight)
        bp = [int(x) for x in c.source_heldout_bp]
        # held-out flags, then each stream's kept documents in shuffled order
        for j in range(J):
            b, e = sdb[j], sdb[j + 1]
            perm = Permutation(e - b, doc_keys(self.seed, j)) if e > b else None
            kept = []
            for p in range(e - b):
                d = b + perm(p)
                if lengths[d] == 0:
                    continue
                rate = bp[ssrc[j]]
                ho = rate > 0 and held_out(text_hash(toks[offs[d]:offs[d + 1]], self.hash_key), rate)
                if ho == self.heldout_only:
                    kept.append(d)
            pack = pack_wrap if self.wrap else pack_greedy
            self.windows.append(pack(kept, lengths, self.T))
        # quotas, the rule restarting at every schedule piece
        pieces = self._pieces()
        self.cum = [[0] * J]
        src_before, str_before = [0] * S, [0] * J
        for k in range(self.K):
            pi = max(i for i, p in enumerate(pieces) if p["begin"] <= k)
            p = pieces[pi]
            if p["begin"] == k:
                src_before, str_before = [0] * S, [0] * J
            n = p["B"]
            a_src = apportion(n, (k - p["begin"] + 1) * n, [int(x) for x in p["source_weight"]],
                              src_before)
            a = [0] * J
            for s in range(S):
                js = [j for j in range(J) if ssrc[j] == s]
                got = apportion(a_src[s], src_before[s] + a_src[s],
                                [int(p["stream_weight"][j]) for j in js],
                                [str_before[j] for j in js])
                for j, g in zip(js, got):
                    a[j] = g
                    str_before[j] += g
                src_before[s] += a_src[s]
            self.quota.append(a)
            self.cum.append([x + y for x, y in zip(self.cum[-1], a)])
        # the first update asking a stream for a window it lacks
        self.valid_steps = self.K
        for k in range(self.K):
            if any(self.cum[k + 1][j] > len(self.windows[j]) for j in range(J)):
                self.valid_steps = k + 1 if self.drain else k
                break
        return self

    # -- reading order ---------------------------------------------------------
    def window_of_rank(self, j, r):
        G, W = self.window_segment, len(self.windows[j])
        if G == 0:
            return r
        s = r // G
        first = s * G
        return first + Permutation(min(G, W - first), segment_keys(self.seed, j, s))(r - first)

    def rows(self, k):
        c = self.corpus
        offs = [int(x) for x in c.doc_offsets]
        T, J = self.T, len(self.windows)
        Bk = self.rows_of(k)
        rho = Permutation(Bk, row_keys(self.seed, k)) if self.shuffle_rows else (lambda i: i)
        out = dict(tokens=[], pos=[], doc=[], mask=[], row_fp=[], row_learned=[], row_len=[])
        for slot in range(Bk):
            i = rho(slot)
            j, first = 0, 0
            while i >= first + self.quota[k][j]:
                first += self.quota[k][j]
                j += 1
            r = self.cum[k][j] + i - first
            tok, pos, doc, msk = [], [], [], []
            if r < len(self.windows[j]):
                for pc in self.windows[j][self.window_of_rank(j, r)]:
                    ls = int(c.loss_start[pc.doc]) if c.loss_start is not None else 0
                    for e in range(pc.length):
                        tok.append(int(c.tokens[offs[pc.doc] + pc.off + e]))
                        pos.append(e)
                        doc.append(pc.doc)
                        msk.append(1 if pc.off + e >= ls else 0)
            real = len(tok)
            pad = T - real
            tok += [self.pad_id] * pad
            pos += [0] * pad
            doc += [-1] * pad
            msk += [0] * pad
            fp = 0
            for t in range(T):
                a = (u32(tok[t]) << 32) | u32(doc[t])
                b = (msk[t] << 32) | u32(pos[t])
                fp = (fp + mix(a ^ (((b | (t << 40)) * GOLDEN) & M64))) & M64
            length = real
            if self.len_bucket:
                length = min(-(-real // self.len_bucket) * self.len_bucket, T)
            for key, v in (("tokens", tok), ("pos", pos), ("doc", doc), ("mask", msk)):
                out[key].append(v)
            out["row_fp"].append(mix(fp))
            out["row_learned"].append(sum(msk))
            out["row_len"].append(length)
        return out

    # -- the order digest ------------------------------------------------------
    def digest(self):
        c = self.corpus
        items = [self.T, self.B, self.K, self.valid_steps,
                 int(self.drain) | int(self.heldout_only) << 1 | int(self.shuffle_rows) << 2
                 | int(self.wrap) << 3,
                 u32(self.pad_id), self.seed & M64, self.hash_key & M64, len(c.source_weight),
                 len(c.stream_source), self.window_segment, self.len_bucket]
        for s in range(len(c.source_weight)):
            items += [int(c.source_weight[s]), int(c.source_heldout_bp[s])]
        for j in range(len(c.stream_source)):
            items += [int(c.stream_doc_begin[j]), int(c.stream_doc_begin[j + 1]),
                      int(c.stream_source[j]), int(c.stream_weight[j])]
        if self.schedule:
            items.append(len(self.schedule))
            for p in self.schedule:
                items += [p["begin"], p["B"]] + [int(x) for x in p["source_weight"]] \
                    + [int(x) for x in p["stream_weight"]]
        for k in range(self.valid_steps):
            items += self.quota[k]
        for j, ws in enumerate(self.windows):
            for r in range(min(self.cum[self.valid_steps][j], len(ws))):
                pc = ws[self.window_of_rank(j, r)][0]
                items.append((pc.doc << 32) | pc.off)
        total = 0
        for n, x in enumerate(items):
            total = (total + mix((x & M64) ^ mix(n))) & M64
        return mix(total ^ len(items))


def twin(corpus, *, seed=None, hash_key=None, T=None, B=None, max_steps=None, drain=None,
         pad_id=None, **options) -> Twin:
    c = corpus
    return Twin(corpus=c, seed=int(c.seed if seed is None else seed) & M64,
                hash_key=int(c.hash_key if hash_key is None else hash_key) & M64,
                T=int(c.T if T is None else T), B=int(c.B if B is None else B),
                K=int(c.max_steps if max_steps is None else max_steps),
                drain=bool(c.drain if drain is None else drain),
                pad_id=int(c.pad_id if pad_id is None else pad_id), **options).build()
