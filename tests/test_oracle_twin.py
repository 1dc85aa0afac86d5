"""The C oracle against an independent pure-Python statement of the same
definitions (``_pytwin.py``), byte for byte on small random corpora, with
every option: held-out rates, completion masks, drain, the validation stream,
windows read in segments, shuffled rows, wrap packing, bucketed row lengths
and schedules."""
import numpy as np
import pytest

import oracle
from _helpers import corpus_from_lengths
from _pytwin import mix, twin


def test_twin_mix_matches_the_oracle():
    rng = np.random.default_rng(0)
    for x in [0, 1, (1 << 64) - 1] + [int(v) for v in rng.integers(0, 2**63, size=50)]:
        assert mix(x) == oracle.splitmix64(x)


def _case(rng):
    T = int(rng.choice([16, 32, 48, 80]))
    J = int(rng.integers(1, 5))
    stream_docs = [int(rng.integers(0, 90)) for _ in range(J)]
    lengths = []
    for _ in range(sum(stream_docs)):
        u = rng.random()
        if u < 0.08:
            lengths.append(0)
        elif u < 0.15:
            lengths.append(T * int(rng.integers(1, 3)))
        elif u < 0.8:
            lengths.append(int(rng.integers(1, T + 1)))
        else:
            lengths.append(int(rng.integers(T, 4 * T)))
    S = int(rng.integers(1, J + 1))
    stream_source = sorted(list(range(S)) + [int(x) for x in rng.integers(0, S, size=J - S)])
    loss_start = None
    if rng.random() < 0.5:
        loss_start = [int(rng.integers(-2, max(L, 1) + 3)) for L in lengths]
    B = int(rng.integers(1, 8))
    K = int(rng.integers(1, 25))
    c = corpus_from_lengths(
        lengths, T=T, B=B, max_steps=K, stream_docs=stream_docs, stream_source=stream_source,
        source_weight=[int(x) for x in rng.integers(1, 9, size=S)],
        stream_weight=[int(x) for x in rng.integers(1, 9, size=J)],
        heldout_bp=[int(rng.choice([0, 500, 3000, 10000])) for _ in range(S)],
        loss_start=loss_start, seed=int(rng.integers(0, 2**63)),
        hash_key=int(rng.integers(0, 2**63)), drain=bool(rng.integers(0, 2)),
        pad_id=int(rng.integers(-3, 1000)))
    opts = dict(heldout_only=bool(rng.random() < 0.25),
                window_segment=int(rng.choice([0, 0, 1, 2, 3, 7])),
                shuffle_rows=bool(rng.integers(0, 2)), wrap=bool(rng.integers(0, 2)),
                len_bucket=int(rng.choice([0, 0, 1, 16, 24])))
    if K >= 3 and rng.random() < 0.4:
        n_p = int(rng.integers(2, min(4, K) + 1))
        begins = [0] + sorted(int(x) for x in rng.choice(np.arange(1, K), size=n_p - 1,
                                                          replace=False))
        opts["schedule"] = [dict(begin=b, B=int(rng.integers(1, B + 1)),
                                 source_weight=[int(x) for x in rng.integers(1, 50, size=S)],
                                 stream_weight=[int(x) for x in rng.integers(1, 50, size=J)])
                            for b in begins]
    return c, opts


@pytest.mark.parametrize("case", range(120))
def test_twin_agrees_with_the_oracle(case):
    rng = np.random.default_rng(31000 + case)
    c, opts = _case(rng)
    o = oracle.Oracle(c, **opts)
    t = twin(c, **opts)
    assert o.valid_steps == t.valid_steps
    q, cum, _ = o.quota()
    assert (q == np.asarray(t.quota, np.int64).reshape(q.shape)).all()
    assert (cum == np.asarray(t.cum, np.int64).reshape(cum.shape)).all()
    for j in range(c.n_streams):
        assert o.n_windows(j) == len(t.windows[j]), j
    assert o.digest == t.digest()
    for k in range(o.valid_steps):
        want = t.rows(k)
        got = o.rows(k)
        for f in ("tokens", "pos", "doc", "mask", "row_fp", "row_learned", "row_len"):
            g = np.asarray(got[f]).astype(np.int64) if f != "row_fp" else got[f]
            w = np.asarray(want[f], dtype=np.uint64 if f == "row_fp" else np.int64)
            assert g.shape == w.shape, (k, f)
            assert (g == w).all(), (k, f)
