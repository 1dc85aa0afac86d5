"""Small hand-built corpora for the tests (no method arithmetic here)."""
import json
import os

import numpy as np

from corpus import Corpus

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def corpus_from_lengths(lengths, *, T, B, max_steps, stream_docs=None, stream_source=None,
                        source_weight=None, stream_weight=None, heldout_bp=None,
                        tokens=None, loss_start=None, seed=0, hash_key=0, drain=False,
                        pad_id=0, name="hand"):
    """A corpus whose document d has ``lengths[d]`` tokens.  Unless given,
    token values encode (doc, offset) as ``doc * 100000 + offset`` so that a
    test can read back where every output token came from."""
    lengths = np.asarray(lengths, dtype=np.int64)
    offs = np.zeros(lengths.size + 1, np.int64)
    np.cumsum(lengths, out=offs[1:])
    if tokens is None:
        tokens = np.concatenate([d * 100000 + np.arange(L, dtype=np.int64)
                                 for d, L in enumerate(lengths)] or [np.zeros(0, np.int64)])
        tokens = tokens.astype(np.int32)
    if stream_docs is None:
        stream_docs = [lengths.size]
    J = len(stream_docs)
    if stream_source is None:
        stream_source = list(range(J))
    S = max(stream_source) + 1
    if source_weight is None:
        source_weight = [1] * S
    if stream_weight is None:
        stream_weight = [1] * J
    if heldout_bp is None:
        heldout_bp = [0] * S
    sdb = np.zeros(J + 1, np.uint32)
    sdb[1:] = np.cumsum(stream_docs)
    return Corpus(name=name, tokens=np.asarray(tokens, np.int32), doc_offsets=offs,
                  loss_start=None if loss_start is None else np.asarray(loss_start, np.int32),
                  stream_doc_begin=sdb, stream_source=np.asarray(stream_source, np.uint32),
                  source_weight=np.asarray(source_weight, np.uint32),
                  stream_weight=np.asarray(stream_weight, np.uint32),
                  source_heldout_bp=np.asarray(heldout_bp, np.uint16),
                  T=T, B=B, max_steps=max_steps, drain=drain, pad_id=pad_id, seed=seed,
                  hash_key=hash_key)
