"""Pins of the packing variants: "wrap" packing (Zephon's pipeline example,
pack_flat with algorithm "wrap": concatenate and cut into rows of exactly T
tokens, across document ends) and row lengths rounded up to a bucket (Linnet
training docs, Other trainers: packed lengths round up to a multiple of the
bucket)."""
import numpy as np
import pytest

import oracle
from _helpers import corpus_from_lengths
from corpus import make_preset


@pytest.mark.parametrize("case", range(10))
def test_wrap_windows_are_consecutive_cuts(case):
    rng = np.random.default_rng(40 + case)
    T = int(rng.choice([16, 32, 64]))
    lengths = [int(x) for x in rng.integers(0, 3 * T, size=int(rng.integers(5, 80)))]
    c = corpus_from_lengths(lengths, T=T, B=int(rng.integers(1, 4)), max_steps=100000,
                            heldout_bp=[3000], drain=True, seed=int(rng.integers(0, 99)))
    o = oracle.Oracle(c, wrap=True)
    held, _ = o.heldout()
    order = [oracle.feistel_pi(c.seed, 0, c.n_docs, p) for p in range(c.n_docs)]
    kept = [d for d in order if lengths[d] > 0 and not held[d]]
    run = np.concatenate([c.tokens[c.doc_offsets[d]:c.doc_offsets[d + 1]] for d in kept]
                         or [np.zeros(0, np.int32)])
    doc, off, ln = o.pieces(0)
    first = o.window_first(0)
    W = first.size - 1
    assert W == -(-run.size // T)
    for r in range(W):
        used = int(ln[first[r]:first[r + 1]].sum())
        assert used == (T if r < W - 1 else run.size - T * (W - 1))
    # the rows of a full pass read the run in order (one stream: rank order)
    got = []
    for k in range(o.valid_steps):
        rr = o.rows(k)
        for i in range(rr["tokens"].shape[0]):
            m = rr["doc"][i] >= 0
            got.append(rr["tokens"][i][m])
            # position ids restart at every piece, the mask follows the
            # in-document offset (every token learned here)
            assert (rr["pos"][i][m] < T).all() and (rr["mask"][i][m] == 1).all()
            assert rr["row_len"][i] == m.sum()
    got = np.concatenate(got) if got else np.zeros(0, np.int32)
    assert np.array_equal(got, run[:got.size])
    assert got.size == run.size or o.valid_steps * c.B * T > got.size


def test_wrap_piece_that_continues_a_document():
    # T = 8, documents of 5, 6, 7 tokens in visit order: 5|3 + 3|... cuts
    T = 8
    n = 3
    order = [oracle.feistel_pi(0, 0, n, p) for p in range(n)]
    lengths = [0] * n
    for p, L in enumerate([5, 6, 7]):
        lengths[order[p]] = L
    c = corpus_from_lengths(lengths, T=T, B=1, max_steps=3)
    o = oracle.Oracle(c, wrap=True)
    doc, off, ln = o.pieces(0)
    assert list(zip(off.tolist(), ln.tolist())) == [(0, 5), (0, 3), (3, 3), (0, 5), (5, 2)]
    assert o.window_first(0).tolist() == [0, 2, 4, 5]
    r1 = o.rows(1)
    assert r1["pos"][0].tolist() == [0, 1, 2, 0, 1, 2, 3, 4]      # 3 of doc 1, 5 of doc 2
    assert r1["tokens"][0][0] == order[1] * 100000 + 3            # doc 1 from offset 3
    r2 = o.rows(2)
    assert r2["pos"][0].tolist() == [0, 1, 0, 0, 0, 0, 0, 0] and r2["row_len"][0] == 2


def test_wrap_mask_uses_the_in_document_offset():
    c = make_preset("c2s")
    o = oracle.Oracle(c, wrap=True)
    doc, off, ln = o.pieces(0)
    # learned positions of a window: per piece, the in-document offsets at or
    # past the document's loss start (a piece may start inside its document)
    first = o.window_first(0)
    r = o.rows(0)
    for i in range(c.B):
        q0, q1 = int(first[i]), int(first[i + 1])
        want = sum(max(0, min(int(off[q]) + int(ln[q]), 10**9) - max(int(off[q]), int(c.loss_start[doc[q]])))
                   for q in range(q0, q1))
        assert r["row_learned"][i] == want


@pytest.mark.parametrize("bucket", [0, 1, 16, 256, 5000])
def test_row_length_bucket(bucket):
    c = make_preset("c1")
    o = oracle.Oracle(c, len_bucket=bucket)
    r = o.rows(0)
    real = (r["doc"] >= 0).sum(1)
    want = real if bucket == 0 else np.minimum(-(-real // bucket) * bucket, c.T)
    assert (r["row_len"] == want).all()
