"""Pins of the read order: each source's windows of a segment are read in a
random order, and the rows of an update may be shuffled (NeuronSpark-Trainer
README, Concepts: the trainer reads each source's windows of a segment in a
random order).  Both are permutations: a pass still reads every window once,
an update still holds the same rows."""
import numpy as np
import pytest

import oracle
from _helpers import corpus_from_lengths
from corpus import make_preset


@pytest.mark.parametrize("G", [1, 2, 3, 5, 8, 64])
def test_window_order_permutes_each_segment(G):
    for W in list(range(1, 40)) + [63, 64, 65, 200]:
        ws = [oracle.window_of_rank(7, 2, G, W, r) for r in range(W)]
        assert sorted(ws) == list(range(W))
        for r, w in enumerate(ws):
            assert r // G == w // G  # stays inside its segment
    assert [oracle.window_of_rank(7, 2, 0, 50, r) for r in range(50)] == list(range(50))


def test_window_order_depends_on_seed_stream_segment():
    a = [oracle.window_of_rank(1, 0, 64, 1000, r) for r in range(64)]
    b = [oracle.window_of_rank(2, 0, 64, 1000, r) for r in range(64)]
    c = [oracle.window_of_rank(1, 1, 64, 1000, r) for r in range(64)]
    d = [oracle.window_of_rank(1, 0, 64, 1000, 64 + r) - 64 for r in range(64)]
    assert len({tuple(a), tuple(b), tuple(c), tuple(d)}) == 4


def test_row_order_is_a_permutation():
    for B in (1, 2, 5, 16, 97, 512):
        for k in (0, 3):
            rows = [oracle.row_of_slot(11, k, B, i) for i in range(B)]
            assert sorted(rows) == list(range(B))
    assert ([oracle.row_of_slot(11, 0, 64, i) for i in range(64)] !=
            [oracle.row_of_slot(11, 1, 64, i) for i in range(64)])


def test_shuffled_windows_full_pass_reads_every_window_once():
    rng = np.random.default_rng(3)
    lengths = [int(x) for x in rng.integers(1, 90, size=300)]
    c = corpus_from_lengths(lengths, T=64, B=3, max_steps=10000, drain=True)
    plain = oracle.Oracle(c)
    shuf = oracle.Oracle(c, window_segment=5)
    assert plain.valid_steps == shuf.valid_steps
    seen_p, seen_s = [], []
    for k in range(plain.valid_steps):
        seen_p += [tuple(r) for r in plain.rows(k)["tokens"]]
        seen_s += [tuple(r) for r in shuf.rows(k)["tokens"]]
    assert sorted(seen_p) == sorted(seen_s)
    assert seen_p != seen_s
    assert plain.digest != shuf.digest


def test_shuffled_rows_hold_the_same_rows():
    c = make_preset("c3s")
    plain = oracle.Oracle(c)
    shuf = oracle.Oracle(c, shuffle_rows=True)
    for k in (0, 5, plain.valid_steps - 1):
        p = plain.rows(k)
        s = shuf.rows(k)
        rho = [oracle.row_of_slot(c.seed, k, c.B, i) for i in range(c.B)]
        for key in p:
            assert np.array_equal(s[key], p[key][rho])
        # slicing still gives the same bytes
        half = [shuf.rows(k, 0, c.B // 2), shuf.rows(k, c.B // 2, c.B)]
        for key in s:
            assert np.array_equal(np.concatenate([h[key] for h in half]), s[key])
    assert plain.digest != shuf.digest
