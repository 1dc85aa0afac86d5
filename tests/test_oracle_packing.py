"""Pins of the oracle's packing and assembly.

Greedy packing cut at document ends (NeuronSpark-Trainer README, Concepts),
rows of exactly T positions padded at the end (Linnet training docs,
Supervised fine-tuning), a position id of 0 at every sequence start (Linnet,
Other trainers), every kept token trained exactly once (max_epochs 1).

A partition of the piece sequence into consecutive windows that each fit in T
and are each maximal (the next piece would not fit) is exactly the greedy
packing, so the brute-force checks below pin it without re-running it.
"""
import numpy as np
import pytest

import oracle
from _helpers import corpus_from_lengths, golden
from corpus import make_preset


def _visit_order(seed, stream, n):
    return [oracle.feistel_pi(seed, stream, n, p) for p in range(n)]


def test_worked_packing_example():
    g = golden("packing_example.json")
    T, lens = g["T"], g["doc_lengths_in_visit_order"]
    n = len(lens)
    order = _visit_order(0, 0, n)
    lengths = [0] * n
    for p, d in enumerate(order):
        lengths[d] = lens[p]
    c = corpus_from_lengths(lengths, T=T, B=1, max_steps=len(g["windows"]))
    o = oracle.Oracle(c)
    doc, off, ln = o.pieces(0)
    want = [(order[v], a, b) for v, a, b in g["pieces"]]
    assert list(zip(doc.tolist(), off.tolist(), ln.tolist())) == want
    assert o.window_first(0).tolist() == g["window_first_piece"] + [len(want)]
    assert np.concatenate([[0], np.cumsum(ln)]).tolist() == g["piece_prefix"]
    assert o.valid_steps == len(g["windows"])
    for k, w in enumerate(g["windows"]):
        r = o.rows(k)
        vis = w["visit"]
        exp_doc = [order[v] if v >= 0 else -1 for v in vis]
        assert r["doc"][0].tolist() == exp_doc
        assert r["pos"][0].tolist() == w["pos"]
        exp_tok = [order[v] * 100000 + od if v >= 0 else 0
                   for v, od in zip(vis, g["window_offset_in_doc"][k])]
        assert r["tokens"][0].tolist() == exp_tok
        assert r["mask"][0].tolist() == [1 if v >= 0 else 0 for v in vis]
        assert r["row_learned"][0] == sum(1 for v in vis if v >= 0)


def _random_case(rng, T):
    J = int(rng.integers(1, 4))
    stream_docs = [int(rng.integers(0, 40)) for _ in range(J)]
    n = sum(stream_docs)
    # a length mix with empty documents, short ones and ones several T long
    lengths = []
    for _ in range(n):
        u = rng.random()
        if u < 0.08:
            lengths.append(0)
        elif u < 0.8:
            lengths.append(int(rng.integers(1, T + 1)))
        else:
            lengths.append(int(rng.integers(T, 4 * T + 1)))
    bp = [int(rng.choice([0, 1500, 5000]))] * J
    return corpus_from_lengths(lengths, T=T, B=max(1, J), max_steps=1, stream_docs=stream_docs,
                               heldout_bp=bp, seed=int(rng.integers(0, 2**62)))


@pytest.mark.parametrize("case", range(40))
def test_packing_brute_force_properties(case):
    rng = np.random.default_rng(100 + case)
    T = int(rng.choice([16, 32, 48]))
    c = _random_case(rng, T)
    o = oracle.Oracle(c)
    held, _ = o.heldout()
    offs = c.doc_offsets
    for j in range(c.n_streams):
        d0, d1 = int(c.stream_doc_begin[j]), int(c.stream_doc_begin[j + 1])
        order = [d0 + x for x in _visit_order(c.seed, j, d1 - d0)]
        kept = [d for d in order if offs[d + 1] > offs[d] and not held[d]]
        doc, off, ln = o.pieces(j)
        # pieces: the kept documents in visit order, each cut into T-chunks
        i = 0
        for d in kept:
            L = int(offs[d + 1] - offs[d])
            for o0 in range(0, L, T):
                assert (doc[i], off[i], ln[i]) == (d, o0, min(T, L - o0))
                i += 1
        assert i == doc.size
        # windows: consecutive, each fits, each maximal (greedy)
        first = o.window_first(j).tolist()
        assert first[0] == 0 and first[-1] == doc.size
        assert all(a < b for a, b in zip(first, first[1:]))
        for r in range(len(first) - 1):
            used = int(ln[first[r]:first[r + 1]].sum())
            assert used <= T
            if r + 1 < len(first) - 1:
                assert used + int(ln[first[r + 1]]) > T
        # a document crosses a window end only as T-chunks: every piece that
        # is not a whole T-chunk sits inside one window with all of its doc's
        # short pieces
        win_of = np.zeros(doc.size, np.int64)
        for r in range(len(first) - 1):
            win_of[first[r]:first[r + 1]] = r
        for q in range(doc.size):
            if ln[q] == T:
                assert first.count(q) == 1 and (q + 1 == doc.size or first.count(q + 1) == 1)


def _full_pass(c):
    """Run every valid update of a drained single-stream recipe."""
    o = oracle.Oracle(c, drain=True)
    rows = [o.rows(k) for k in range(o.valid_steps)]
    return o, rows


@pytest.mark.parametrize("case", range(12))
def test_every_kept_token_exactly_once(case):
    rng = np.random.default_rng(500 + case)
    T = int(rng.choice([16, 64]))
    n = int(rng.integers(5, 120))
    lengths = [int(x) for x in rng.integers(0, 3 * T, size=n)]
    B = int(rng.integers(1, 5))
    c = corpus_from_lengths(lengths, T=T, B=B, max_steps=10000, heldout_bp=[2000],
                            seed=int(rng.integers(0, 1000)))
    o, rows = _full_pass(c)
    held, _ = o.heldout()
    seen = {}
    for k, r in enumerate(rows):
        real = r["doc"] >= 0
        # position ids restart at 0 at every piece start and stay below T
        assert (r["pos"] >= 0).all() and (r["pos"] < T).all()
        assert (r["mask"][~real] == 0).all() and (r["pos"][~real] == 0).all()
        assert (r["tokens"][~real] == c.pad_id).all()
        for d, t in zip(r["doc"][real].tolist(), r["tokens"][real].tolist()):
            assert t // 100000 == d
            key = (d, t % 100000)
            assert key not in seen, key
            seen[key] = k
        # padding only at the end of a row
        for row in real:
            nz = np.flatnonzero(row)
            if nz.size:
                assert nz[-1] == nz.size - 1
    want = {(d, x) for d in range(n) if not held[d] for x in range(lengths[d])}
    assert set(seen) == want
    # the final update is the drained one: it may hold rows that learn nothing
    assert o.valid_steps >= 1
    assert all(r["row_learned"].min() > 0 for r in rows[:-1])


def test_sft_completion_only_mask():
    c = make_preset("c2s")
    o = oracle.Oracle(c)
    for k in range(min(4, o.valid_steps)):
        r = o.rows(k)
        real = r["doc"] >= 0
        ls = c.loss_start[np.where(real, r["doc"], 0)]
        # examples are at most T long, so the in-document offset is pos
        assert ((r["mask"] == 1) == (real & (r["pos"] >= ls))).all()
        assert (r["row_learned"] == r["mask"].sum(1)).all()
        assert (r["row_learned"] < real.sum(1)).all()  # prompts are never learned


def test_long_documents_cut_into_t_chunks():
    c = make_preset("c5s")
    o = oracle.Oracle(c)
    T = c.T
    doc, off, ln = o.pieces(0)
    full = ln == T
    assert full.any()
    first = o.window_first(0)
    # a full chunk is its own window
    for q in np.flatnonzero(full)[:200]:
        r = int(np.searchsorted(first, q, side="right") - 1)
        assert first[r] == q and first[r + 1] == q + 1
    # and reads as one sequence 0..T-1 of one document
    k_seen = 0
    for k in range(min(o.valid_steps, 8)):
        r = o.rows(k)
        for i in range(c.B):
            if r["pos"][i, -1] == T - 1:
                assert (r["pos"][i] == np.arange(T)).all()
                assert (r["doc"][i] == r["doc"][i, 0]).all()
                k_seen += 1
    assert k_seen > 0
