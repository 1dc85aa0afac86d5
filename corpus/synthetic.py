"""Seeded synthetic corpora shaped like the workloads of the packed-assembly path.

Every array is drawn with numpy's PCG64 from a ``SeedSequence`` keyed by a
data seed, so a corpus is a pure function of its parameters.  Token ids are
drawn in fixed-size chunks, each from its own child sequence, so the result
does not depend on how many threads fill it.

Shapes (document-length mixes, vocabularies, mixtures of sources and strata)
follow the workloads named for this path:

* pretraining mixtures: document lengths ``clip(rint(median * exp(sigma * z)),
  lo, hi)`` with ``z`` standard normal, token ids uniform in ``[0, vocab)``;
* SFT examples: a prompt and a completion, each log-normal, whose first
  ``prompt`` positions are not learned (the ``loss_start`` array);
* a long-context corpus drawn document by document until a token budget is
  reached.

No dataset is read: these arrays stand in for the web corpora the workloads
were quoted on.  Nothing here computes a hash, a permutation, a quota or a
packing; that is the method, and it lives elsewhere.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

TOKEN_CHUNK = 1 << 22  # tokens per independently seeded chunk


@dataclass
class Corpus:
    """One synthetic corpus plus the packing recipe that goes with it."""

    name: str
    tokens: np.ndarray            # int32 [n_tokens]
    doc_offsets: np.ndarray       # int64 [n_docs + 1], nondecreasing, [0] == 0
    loss_start: Optional[np.ndarray]  # int32 [n_docs] or None (every token learned)
    stream_doc_begin: np.ndarray  # uint32 [n_streams + 1]
    stream_source: np.ndarray     # uint32 [n_streams], nondecreasing
    source_weight: np.ndarray     # uint32 [n_sources], > 0
    stream_weight: np.ndarray     # uint32 [n_streams], > 0
    source_heldout_bp: np.ndarray  # uint16 [n_sources], 0..10000
    T: int
    B: int
    max_steps: int
    drain: bool = False
    pad_id: int = 0
    seed: int = 0
    hash_key: int = 0
    vocab: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def n_docs(self) -> int:
        return int(self.doc_offsets.shape[0] - 1)

    @property
    def n_tokens(self) -> int:
        return int(self.tokens.shape[0])

    @property
    def n_streams(self) -> int:
        return int(self.stream_source.shape[0])

    @property
    def n_sources(self) -> int:
        return int(self.source_weight.shape[0])

    def recipe(self) -> dict:
        """The scalar part of the packing recipe (for logs and configs)."""
        return dict(name=self.name, n_docs=self.n_docs, n_tokens=self.n_tokens,
                    n_sources=self.n_sources, n_streams=self.n_streams, T=self.T,
                    B=self.B, max_steps=self.max_steps, drain=self.drain,
                    seed=self.seed, hash_key=self.hash_key, pad_id=self.pad_id,
                    vocab=self.vocab)


def _lognormal_lengths(z: np.ndarray, median: float, sigma: float, lo: int,
                       hi: Optional[int]) -> np.ndarray:
    x = np.rint(median * np.exp(sigma * z))
    x = np.maximum(x, lo)
    if hi is not None:
        x = np.minimum(x, hi)
    return x.astype(np.int64)


def _fill_tokens(ss: np.random.SeedSequence, n_tokens: int, vocab: int,
                 threads: Optional[int] = None) -> np.ndarray:
    out = np.empty(n_tokens, dtype=np.int32)
    n_chunks = (n_tokens + TOKEN_CHUNK - 1) // TOKEN_CHUNK
    children = ss.spawn(n_chunks)

    def fill(c: int) -> None:
        lo = c * TOKEN_CHUNK
        hi = min(n_tokens, lo + TOKEN_CHUNK)
        g = np.random.Generator(np.random.PCG64(children[c]))
        out[lo:hi] = g.integers(0, vocab, size=hi - lo, dtype=np.int32)

    if threads is None:
        threads = min(32, os.cpu_count() or 1)
    if n_chunks <= 1 or threads <= 1:
        for c in range(n_chunks):
            fill(c)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out


def _split_docs(total: int, parts: list[int]) -> list[int]:
    """Document counts per stream proportional to ``parts``: floor of each
    proportional share, the rounding remainder going to the last stream."""
    P = sum(parts)
    counts = [total * p // P for p in parts]
    counts[-1] += total - sum(counts)
    return counts


def make_corpus(name: str, *, data_seed: int, vocab: int, T: int, B: int,
                max_steps: int, source_weight: list[int], stream_source: list[int],
                stream_weight: list[int], heldout_bp: list[int],
                stream_docs: Optional[list[int]] = None,
                target_tokens: Optional[int] = None,
                length: tuple = (200.0, 1.0, 1, 8192),
                sft: Optional[dict] = None, drain: bool = False, seed: int = 0,
                hash_key: int = 0, pad_id: int = 0,
                threads: Optional[int] = None) -> Corpus:
    """Draw one corpus.

    ``stream_docs`` gives the document count of every stream (documents are
    laid out stream after stream); alternatively ``target_tokens`` (single
    stream only) draws documents until their total length reaches the target.
    ``length`` is ``(median, sigma, lo, hi)`` (``hi`` may be None).  ``sft``
    (``dict(prompt_median, completion_median, sigma, max_total)``) draws
    prompt/completion examples instead and sets ``loss_start`` to the prompt
    length.
    """
    ss = np.random.SeedSequence(data_seed)
    len_ss, tok_ss = ss.spawn(2)
    lg = np.random.Generator(np.random.PCG64(len_ss))
    loss_start = None
    if target_tokens is not None:
        assert len(stream_source) == 1, "target_tokens is for one stream"
        median, sigma, lo, hi = length
        chunks, total = [], 0
        while total < target_tokens:
            ln = _lognormal_lengths(lg.standard_normal(1 << 16), median, sigma, lo, hi)
            cs = np.cumsum(ln)
            if total + int(cs[-1]) >= target_tokens:
                k = int(np.searchsorted(cs, target_tokens - total, side="left"))
                ln = ln[:k + 1]
            chunks.append(ln)
            total += int(ln.sum())
        lengths = np.concatenate(chunks)
        stream_docs = [int(lengths.shape[0])]
    else:
        assert stream_docs is not None
        n_docs = int(sum(stream_docs))
        if sft is not None:
            zp = lg.standard_normal(n_docs)
            zc = lg.standard_normal(n_docs)
            mt = int(sft["max_total"])
            p = _lognormal_lengths(zp, sft["prompt_median"], sft["sigma"], 1, mt - 1)
            c = _lognormal_lengths(zc, sft["completion_median"], sft["sigma"], 1, None)
            over = p + c > mt
            c = np.where(over, np.maximum(1, mt - p), c)
            lengths = p + c
            loss_start = p.astype(np.int32)
        else:
            median, sigma, lo, hi = length
            lengths = _lognormal_lengths(lg.standard_normal(n_docs), median, sigma, lo, hi)
    doc_offsets = np.zeros(lengths.shape[0] + 1, dtype=np.int64)
    np.cumsum(lengths, out=doc_offsets[1:])
    n_tokens = int(doc_offsets[-1])
    tokens = _fill_tokens(tok_ss, n_tokens, vocab, threads)
    sdb = np.zeros(len(stream_docs) + 1, dtype=np.uint32)
    sdb[1:] = np.cumsum(np.asarray(stream_docs, dtype=np.uint64)).astype(np.uint32)
    return Corpus(
        name=name, tokens=tokens, doc_offsets=doc_offsets, loss_start=loss_start,
        stream_doc_begin=sdb,
        stream_source=np.asarray(stream_source, dtype=np.uint32),
        source_weight=np.asarray(source_weight, dtype=np.uint32),
        stream_weight=np.asarray(stream_weight, dtype=np.uint32),
        source_heldout_bp=np.asarray(heldout_bp, dtype=np.uint16),
        T=T, B=B, max_steps=max_steps, drain=drain, pad_id=pad_id, seed=seed,
        hash_key=hash_key, vocab=vocab,
        notes=dict(data_seed=data_seed, length=length, sft=sft,
                   target_tokens=target_tokens))


def _dirichlet_mixture(n_sources: int, n_strata: int, share_seed: int = 1):
    """Integer source and stratum weights from Dirichlet(1) shares drawn from
    ``default_rng(share_seed)``: sources first, then each source's strata."""
    rng = np.random.default_rng(share_seed)
    src = rng.dirichlet([1.0] * n_sources)
    strata = [rng.dirichlet([1.0] * n_strata) for _ in range(n_sources)]
    w = [max(1, int(np.rint(s * 1e9))) for s in src]
    v = [[max(1, int(np.rint(x * 1e9))) for x in st] for st in strata]
    return w, v


def _mixture_kwargs(n_sources: int, n_strata: int, n_docs: int, bp_default: int,
                    bp_last: int) -> dict:
    w, v = _dirichlet_mixture(n_sources, n_strata)
    stream_source, stream_weight, parts = [], [], []
    for s in range(n_sources):
        for t in range(n_strata):
            stream_source.append(s)
            stream_weight.append(v[s][t])
            parts.append(w[s] * v[s][t])
    bp = [bp_default] * n_sources
    bp[-1] = bp_last
    return dict(source_weight=w, stream_source=stream_source,
                stream_weight=stream_weight, heldout_bp=bp,
                stream_docs=_split_docs(n_docs, parts))


def _preset_kwargs(name: str) -> dict:
    # --- the five workloads at full size --------------------------------
    if name == "c1":   # 2 sources x 5,000 docs, shares 7:3, 1 % held out
        return dict(data_seed=1001, vocab=32000, T=1024, B=16, max_steps=10,
                    source_weight=[7, 3], stream_source=[0, 1], stream_weight=[1, 1],
                    heldout_bp=[100, 100], stream_docs=[5000, 5000],
                    length=(200.0, 1.0, 1, 8192))
    if name == "c2":   # SFT: 200,000 prompt/completion examples
        return dict(data_seed=1002, vocab=128256, T=4096, B=8, max_steps=500,
                    source_weight=[1], stream_source=[0], stream_weight=[1],
                    heldout_bp=[0], stream_docs=[200000],
                    sft=dict(prompt_median=64.0, completion_median=128.0, sigma=1.0,
                             max_total=4096))
    if name == "c3":   # 15 sources x 3 strata, Dirichlet shares, 1 % / 5 % held out
        kw = _mixture_kwargs(15, 3, 2_000_000, 100, 500)
        return dict(data_seed=1003, vocab=64000, T=4096, B=512, max_steps=1000,
                    length=(600.0, 1.2, 1, 65536), **kw)
    if name == "c4":   # elastic-determinism check: 4 equal sources, 8 M docs
        return dict(data_seed=1004, vocab=50257, T=8192, B=256, max_steps=200,
                    source_weight=[1, 1, 1, 1], stream_source=[0, 1, 2, 3],
                    stream_weight=[1, 1, 1, 1], heldout_bp=[0, 0, 0, 0],
                    stream_docs=[2_000_000] * 4, length=(400.0, 1.0, 1, None))
    if name == "c5":   # long context: ~1e9 tokens, T = 32768, full pass
        return dict(data_seed=1005, vocab=151936, T=32768, B=64, max_steps=1024,
                    source_weight=[1], stream_source=[0], stream_weight=[1],
                    heldout_bp=[0], target_tokens=1_000_000_000,
                    length=(2048.0, 1.5, 1, 262144), drain=True)
    # --- a medium cut of c3 (same shape, 1/10 of the documents) for profiles
    if name == "c3m":
        kw = _mixture_kwargs(15, 3, 200_000, 100, 500)
        return dict(data_seed=1013, vocab=64000, T=4096, B=512, max_steps=96,
                    length=(600.0, 1.2, 1, 65536), **kw)
    # --- the same cuts of c4 and c5 (the rows of the full workloads over a
    # tenth of the corpus) for profiles
    if name == "c4m":
        return dict(data_seed=1014, vocab=50257, T=8192, B=256, max_steps=64,
                    source_weight=[1, 1, 1, 1], stream_source=[0, 1, 2, 3],
                    stream_weight=[1, 1, 1, 1], heldout_bp=[0, 0, 0, 0],
                    stream_docs=[200_000] * 4, length=(400.0, 1.0, 1, None))
    if name == "c5m":
        return dict(data_seed=1015, vocab=151936, T=32768, B=64, max_steps=1024,
                    source_weight=[1], stream_source=[0], stream_weight=[1],
                    heldout_bp=[0], target_tokens=100_000_000,
                    length=(2048.0, 1.5, 1, 262144), drain=True)
    # --- shrunk variants with the same structure (CPU-sized) ------------
    if name == "c2s":
        return dict(data_seed=2002, vocab=128256, T=4096, B=8, max_steps=16,
                    source_weight=[1], stream_source=[0], stream_weight=[1],
                    heldout_bp=[0], stream_docs=[2000],
                    sft=dict(prompt_median=64.0, completion_median=128.0, sigma=1.0,
                             max_total=4096))
    if name == "c3s":
        kw = _mixture_kwargs(15, 3, 20_000, 100, 500)
        return dict(data_seed=2003, vocab=64000, T=1024, B=128, max_steps=40,
                    length=(150.0, 1.2, 1, 16384), **kw)
    if name == "c4s":
        return dict(data_seed=2004, vocab=50257, T=2048, B=64, max_steps=30,
                    source_weight=[1, 1, 1, 1], stream_source=[0, 1, 2, 3],
                    stream_weight=[1, 1, 1, 1], heldout_bp=[0, 0, 0, 0],
                    stream_docs=[5000] * 4, length=(100.0, 1.0, 1, None))
    if name == "c5s":
        return dict(data_seed=2005, vocab=151936, T=8192, B=8, max_steps=256,
                    source_weight=[1], stream_source=[0], stream_weight=[1],
                    heldout_bp=[0], target_tokens=4_000_000,
                    length=(512.0, 1.5, 1, 65536), drain=True)
    raise KeyError(name)


PRESETS = ("c1", "c2", "c3", "c4", "c5", "c3m", "c4m", "c5m", "c2s", "c3s", "c4s", "c5s")


def make_preset(name: str, threads: Optional[int] = None, **overrides) -> Corpus:
    """One of the named workloads (``c1``..``c5`` full size, ``c3m``..``c5m``
    a tenth of ``c3``..``c5``, ``c2s``..``c5s`` shrunk with the same
    structure); ``overrides`` replace recipe fields."""
    kw = _preset_kwargs(name)
    kw.update(overrides)
    return make_corpus(name, threads=threads, **kw)
