"""Pins of the oracle's per-update mixture apportionment.

NeuronSpark-Trainer README, Concepts: every update holds each source within
two samples of its recipe share; every stratum of a source is held at its
share.  The rule is checked against a hand-worked example and against an
exhaustive search written as an optimisation (not as the rule): among all
allocations that give each child the floor of its exact share or one more,
the one whose sorted cumulative shortfalls are lexicographically smallest
(ties: the lowest indices get the extra windows).

Per update a child gets at most one window more or less than its exact share
(at most, not strictly less: a child whose exact share is a whole number can
still take an extra window when its cumulative shortfall is the largest), so
no source's count is ever more than two windows off its share.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle
from _helpers import corpus_from_lengths, golden
from corpus.synthetic import _preset_kwargs


def test_worked_quota_example():
    g = golden("quota_example.json")
    v, B = g["weights"], g["B"]
    C = [0] * len(v)
    seq = []
    for k in range(3 * g["period"]):
        a = oracle.apportion(v, C, B, (k + 1) * B)
        seq.append(a)
        C = [c + x for c, x in zip(C, a)]
        if k == 4:
            assert C == g["cumulative_after_update_4"]
    assert seq[:5] == g["updates"]
    p = g["period"]
    assert all(seq[k] == seq[k + p] for k in range(len(seq) - p))


def test_worked_quota_example_through_recipe():
    g = golden("quota_example.json")
    c = corpus_from_lengths([5] * 4, T=16, B=g["B"], max_steps=5, stream_docs=[2, 2],
                            source_weight=g["weights"])
    q, cum, sq = oracle.Oracle(c).quota()
    assert q.tolist() == g["updates"]
    assert sq.tolist() == g["updates"]
    assert cum[5].tolist() == g["cumulative_after_update_4"]


def _brute(v, C, n, N):
    V = sum(v)
    exact = [Fraction(n * x, V) for x in v]
    ideal = [Fraction(N * x, V) for x in v]
    floors = [int(e) for e in exact]
    best = None
    for alloc in itertools.product(*[(f, f + 1) for f in floors]):
        if sum(alloc) != n:
            continue
        short = sorted((ideal[c] - (C[c] + alloc[c]) for c in range(len(v))), reverse=True)
        bumped = tuple(c for c in range(len(v)) if alloc[c] > floors[c])
        key = (short, bumped)
        if best is None or key < best[0]:
            best = (key, list(alloc))
    return best[1]


def test_quota_integer_share_can_take_the_extra_window():
    # weights 4:1:3, 12 windows, shares 6, 1.5, 4.5; cumulative shortfalls
    # before the extra window 4/8, 1/8, 3/8: the source whose exact share is 6
    # takes it (7 windows, one more than its share; still within two).
    assert oracle.apportion([4, 1, 3], [14, 4, 11], 12, 41) == [7, 1, 4]


@pytest.mark.parametrize("case", range(300))
def test_quota_rule_matches_exhaustive_search(case):
    rng = np.random.default_rng(case)
    S = int(rng.integers(1, 6))
    v = [int(x) for x in rng.integers(1, 12, size=S)]
    # a history: run a few updates of random sizes through the rule itself,
    # then check one more against the search
    C = [0] * S
    tot = 0
    for _ in range(int(rng.integers(0, 6))):
        n = int(rng.integers(0, 15))
        tot += n
        a = oracle.apportion(v, C, n, tot)
        C = [c + x for c, x in zip(C, a)]
    n = int(rng.integers(0, 15))
    tot += n
    assert oracle.apportion(v, C, n, tot) == _brute(v, C, n, tot)


def test_quota_invariants_on_dirichlet_mixture():
    kw = _preset_kwargs("c3")
    J = len(kw["stream_source"])
    K, B = 1000, 512
    c = corpus_from_lengths([1] * J, T=16, B=B, max_steps=K, stream_docs=[1] * J,
                            stream_source=kw["stream_source"], source_weight=kw["source_weight"],
                            stream_weight=kw["stream_weight"])
    q, cum, sq = oracle.Oracle(c).quota()
    w = np.asarray(kw["source_weight"], dtype=np.float64)
    V = w.sum()
    assert (q >= 0).all() and (sq >= 0).all()
    assert (sq.sum(1) == B).all()
    # per update, each source within one window of its share (so within two)
    assert (np.abs(sq - B * w[None, :] / V) <= 1).all()
    # cumulatively too: within two windows of the share after every update
    csum = np.cumsum(sq, axis=0)
    k = np.arange(1, K + 1, dtype=np.float64)[:, None]
    assert (np.abs(csum - k * B * w[None, :] / V) < 2).all()
    # strata within their source
    ss = np.asarray(kw["stream_source"])
    sw = np.asarray(kw["stream_weight"], dtype=np.float64)
    for s in range(len(w)):
        js = np.flatnonzero(ss == s)
        Vs = sw[js].sum()
        assert (q[:, js].sum(1) == sq[:, s]).all()
        assert (np.abs(q[:, js] - sq[:, s:s + 1] * sw[None, js] / Vs) <= 1).all()
    assert (cum[1:] == np.cumsum(q, axis=0)).all()


def test_quota_equal_weights_round_robin():
    # four equal sources, 6 windows per update: 2,2,1,1 then 1,1,2,2 ...
    C = [0, 0, 0, 0]
    tot = 0
    for k in range(8):
        tot += 6
        a = oracle.apportion([1, 1, 1, 1], C, 6, tot)
        assert sorted(a) == [1, 1, 2, 2]
        C = [c + x for c, x in zip(C, a)]
        assert max(C) - min(C) <= 1
