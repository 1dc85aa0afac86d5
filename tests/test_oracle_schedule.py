"""Pins of schedules: an append-only mixture schedule and a batch-size ramp
(NeuronSpark-Trainer README, Concepts and Training: the mixture schedule is
append-only; tokens per update follow a ramp of pieces; Zephon: the work
source may change the mixture's weights during a run).  Each piece of the
horizon has its own weights and rows per update; the quota rule starts its
counts again at every piece, while the windows each stream has given run on,
so every row stays a pure function of (seed, update)."""
import numpy as np
import pytest

import oracle
from _helpers import corpus_from_lengths
from corpus.synthetic import _preset_kwargs


def _mixture_corpus(K, B, n_docs_per_stream=400, seed=0):
    kw = _preset_kwargs("c3s")
    J = len(kw["stream_source"])
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(1, 300, size=J * n_docs_per_stream)]
    return corpus_from_lengths(lengths, T=256, B=B, max_steps=K,
                               stream_docs=[n_docs_per_stream] * J,
                               stream_source=kw["stream_source"],
                               source_weight=kw["source_weight"],
                               stream_weight=kw["stream_weight"]), kw


def _schedule(kw, rng, begins, Bs):
    S, J = len(kw["source_weight"]), len(kw["stream_weight"])
    return [dict(begin=b, B=Bk, source_weight=[int(x) for x in rng.integers(1, 1000, size=S)],
                 stream_weight=[int(x) for x in rng.integers(1, 1000, size=J)])
            for b, Bk in zip(begins, Bs)]


def test_one_piece_schedule_is_the_plain_recipe():
    c, kw = _mixture_corpus(20, 64)
    sched = [dict(begin=0, B=64, source_weight=kw["source_weight"],
                  stream_weight=kw["stream_weight"])]
    a, b = oracle.Oracle(c), oracle.Oracle(c, schedule=sched)
    qa, ca, _ = a.quota()
    qb, cb, _ = b.quota()
    assert (qa == qb).all() and (ca == cb).all()
    for k in (0, 7, 19):
        for key, v in a.rows(k).items():
            assert np.array_equal(v, b.rows(k)[key])


def test_each_piece_restarts_the_rule():
    rng = np.random.default_rng(1)
    c, kw = _mixture_corpus(30, 96)
    sched = _schedule(kw, rng, [0, 7, 19], [96, 40, 77])
    q, cum, sq = oracle.Oracle(c, schedule=sched).quota()
    bounds = [0, 7, 19, 30]
    for p, piece in enumerate(sched):
        k0, k1 = bounds[p], bounds[p + 1]
        fresh = corpus_from_lengths(np.diff(c.doc_offsets), T=256, B=piece["B"],
                                    max_steps=k1 - k0,
                                    stream_docs=np.diff(c.stream_doc_begin).tolist(),
                                    stream_source=kw["stream_source"],
                                    source_weight=piece["source_weight"],
                                    stream_weight=piece["stream_weight"])
        fq, _, fsq = oracle.Oracle(fresh).quota()
        assert (q[k0:k1] == fq).all(), p
        assert (sq[k0:k1] == fsq).all(), p
        assert (q[k0:k1].sum(1) == piece["B"]).all()
        w = np.asarray(piece["source_weight"], np.float64)
        assert (np.abs(sq[k0:k1] - piece["B"] * w / w.sum()) <= 1).all()
    # the windows each stream has given run on across pieces
    assert (cum[1:] == np.cumsum(q, axis=0)).all()


def test_batch_ramp_rows_and_a_full_pass():
    rng = np.random.default_rng(2)
    lengths = [int(x) for x in rng.integers(1, 120, size=600)]
    c = corpus_from_lengths(lengths, T=128, B=8, max_steps=100000, drain=True)
    sched = [dict(begin=0, B=2, source_weight=[1], stream_weight=[1]),
             dict(begin=5, B=8, source_weight=[1], stream_weight=[1]),
             dict(begin=9, B=5, source_weight=[1], stream_weight=[1])]
    o = oracle.Oracle(c, schedule=sched)
    plain = oracle.Oracle(c)
    seen = []
    for k in range(o.valid_steps):
        r = o.rows(k)
        assert r["tokens"].shape[0] == o.rows_of_step(k)
        seen += [tuple(x) for x in r["tokens"]]
    # one stream: the ramp reads the same windows, in the same order
    flat = []
    for k in range(plain.valid_steps):
        flat += [tuple(x) for x in plain.rows(k)["tokens"]]
    assert seen[:len(flat) - 8] == flat[:len(flat) - 8]
    with pytest.raises(oracle.OracleError) as e:
        o.rows(0, 0, 3)  # update 0 has 2 rows
    assert e.value.code == oracle.INVALID_ARG


def test_schedule_is_in_the_digest():
    rng = np.random.default_rng(3)
    c, kw = _mixture_corpus(20, 64)
    s1 = _schedule(kw, rng, [0, 10], [64, 32])
    s2 = [dict(s1[0]), dict(s1[1], B=31)]
    assert oracle.Oracle(c, schedule=s1).digest != oracle.Oracle(c, schedule=s2).digest


def test_bad_schedules_are_rejected():
    c, kw = _mixture_corpus(20, 64)
    S, J = len(kw["source_weight"]), len(kw["stream_weight"])
    ok = dict(source_weight=[1] * S, stream_weight=[1] * J)
    for bad in ([dict(ok, begin=1, B=8)],                                  # not from 0
                [dict(ok, begin=0, B=8), dict(ok, begin=0, B=8)],          # not increasing
                [dict(ok, begin=0, B=65)],                                 # above B
                [dict(ok, begin=0, B=8), dict(ok, begin=20, B=8)]):        # past the horizon
        with pytest.raises(oracle.OracleError) as e:
            oracle.Oracle(c, schedule=bad)
        assert e.value.code == oracle.INVALID_ARG
