"""Pins of the validation stream: each source's validation rows come from
the held-out documents of every stratum (NeuronSpark-Trainer README,
Concepts).  Packing the held-out documents must give exactly the complement
of the training stream within the sources that hold out, every held-out token
once."""
import numpy as np

import oracle
from _helpers import corpus_from_lengths
from corpus import make_preset


def _tokens_of_pass(o):
    seen = []
    for k in range(o.valid_steps):
        r = o.rows(k)
        real = r["doc"] >= 0
        seen.extend(zip(r["doc"][real].tolist(), r["pos"][real].tolist(),
                        r["tokens"][real].tolist()))
    return seen


def test_validation_is_the_complement_of_training():
    c = make_preset("c1")
    train = oracle.Oracle(c, drain=True)
    val = oracle.Oracle(c, drain=True, heldout_only=True)
    held, _ = train.heldout()
    lengths = np.diff(c.doc_offsets)
    for j in range(c.n_streams):
        d0, d1 = int(c.stream_doc_begin[j]), int(c.stream_doc_begin[j + 1])
        tdoc, toff, tlen = train.pieces(j)
        vdoc, voff, vlen = val.pieces(j)
        stream = set(range(d0, d1))
        assert set(vdoc.tolist()) == {d for d in stream if held[d] and lengths[d] > 0}
        assert set(tdoc.tolist()) == {d for d in stream if not held[d] and lengths[d] > 0}
        # every held-out token of the stream exactly once
        assert int(vlen.sum()) == int(lengths[d0:d1][held[d0:d1]].sum())
    # the rows of the validation updates come from held-out documents only
    docs = {d for d, _, _ in _tokens_of_pass(val)}
    assert docs and all(held[d] for d in docs)
    assert val.digest != train.digest


def test_validation_of_a_source_without_held_out_rate_is_empty():
    c = corpus_from_lengths([30] * 8, T=32, B=2, max_steps=4, stream_docs=[4, 4],
                            heldout_bp=[10000, 0], drain=True)
    o = oracle.Oracle(c, heldout_only=True)
    assert o.n_windows(0) == 4 and o.n_windows(1) == 0
    assert o.valid_steps == 1  # the second source is dry at once: one drained update
    r = o.rows(0)
    assert (r["doc"][0] >= 0).any() and (r["doc"][1] == -1).all()
