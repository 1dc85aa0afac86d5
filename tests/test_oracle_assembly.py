"""Pins of the oracle's batch assembly, fingerprints and step bookkeeping.

* Zephon blog (checkpoint on 16 GPUs, resume on 8/32/64): a global batch is
  byte-identical however it is computed -- here, however its rows are sliced.
* NeuronSpark-Trainer README, Concepts: max_epochs 1, running out of a
  source is an error rather than another epoch; Training: a resume checks
  the sample order's digest.
* Linnet training docs, Reinforcement learning / JAX: a short last step is
  filled with rows that learn nothing.
"""
import hashlib
import os

import numpy as np
import pytest

import oracle
from _helpers import GOLDEN, corpus_from_lengths
from corpus import make_preset

M64 = (1 << 64) - 1
G = 0x9E3779B97F4A7C15


def _published():
    vals = []
    with open(os.path.join(GOLDEN, "splitmix64_seed0.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                vals.append(int(line.split()[1], 16))
    return vals


def test_batch_fold_reaches_published_outputs():
    out = _published()
    assert oracle.batch_fp(np.zeros(0, np.uint64)) == 0
    # F_1 = splitmix64(0 ^ fp_0); choose fp_i = F_i ^ (i * golden) so that
    # F_{i+1} = splitmix64(i * golden), the (i+1)-th published output.
    fps, F = [0], out[0]
    for i in range(1, len(out)):
        fps.append(F ^ ((i * G) & M64))
        F = out[i]
        assert oracle.batch_fp(np.asarray(fps, dtype=np.uint64)) == F


def _row(rng, T):
    return dict(tokens=rng.integers(0, 60000, size=T).astype(np.int32),
                pos=rng.integers(0, T, size=T).astype(np.int32),
                doc=rng.integers(-1, 1000, size=T).astype(np.int32),
                mask=rng.integers(0, 2, size=T).astype(np.uint8))


def _fp(r):
    return oracle.row_fp(r["tokens"], r["pos"], r["doc"], r["mask"])


def _unmix(y):
    from test_oracle_pins import _splitmix_inverse
    return _splitmix_inverse(y)


def test_row_fingerprint_is_a_sum_over_positions_then_one_mix():
    rng = np.random.default_rng(1)
    T = 64
    for _ in range(20):
        r = _row(rng, T)
        base = _unmix(_fp(r))
        t1, t2 = rng.choice(T, size=2, replace=False)
        r1 = {k: v.copy() for k, v in r.items()}
        r1["tokens"][t1] += 1
        r2 = {k: v.copy() for k, v in r.items()}
        r2["mask"][t2] ^= 1
        r12 = {k: v.copy() for k, v in r1.items()}
        r12["mask"][t2] ^= 1
        d1 = (_unmix(_fp(r1)) - base) & M64
        d2 = (_unmix(_fp(r2)) - base) & M64
        assert (_unmix(_fp(r12)) - base) & M64 == (d1 + d2) & M64


def test_row_fingerprint_sees_every_field_and_position():
    rng = np.random.default_rng(2)
    T = 32
    r = _row(rng, T)
    f0 = _fp(r)
    for field in ("tokens", "pos", "doc", "mask"):
        for t in (0, 7, T - 1):
            q = {k: v.copy() for k, v in r.items()}
            q[field][t] = q[field][t] ^ 1
            assert _fp(q) != f0, (field, t)
    # position-keyed: swapping two different positions' contents changes it
    q = {k: v.copy() for k, v in r.items()}
    for k in q:
        q[k][[3, 4]] = q[k][[4, 3]]
    assert _fp(q) != f0
    # token and doc are not interchangeable, nor are mask and pos
    a = dict(tokens=np.full(T, 5, np.int32), pos=np.zeros(T, np.int32),
             doc=np.full(T, 9, np.int32), mask=np.zeros(T, np.uint8))
    b = dict(tokens=np.full(T, 9, np.int32), pos=np.zeros(T, np.int32),
             doc=np.full(T, 5, np.int32), mask=np.zeros(T, np.uint8))
    assert _fp(a) != _fp(b)
    a2 = dict(a, pos=np.ones(T, np.int32), mask=np.zeros(T, np.uint8))
    b2 = dict(a, pos=np.zeros(T, np.int32), mask=np.ones(T, np.uint8))
    assert _fp(a2) != _fp(b2)


@pytest.mark.parametrize("name", ["c1", "c3s"])
def test_rows_identical_under_any_slicing(name):
    c = make_preset(name)
    o = oracle.Oracle(c)
    rng = np.random.default_rng(7)
    for k in range(min(3, o.valid_steps)):
        full = o.rows(k)
        for R in (2, 4, 8):
            if c.B % R:
                continue
            parts = [o.rows(k, i * c.B // R, (i + 1) * c.B // R) for i in range(R)]
            for key in full:
                assert (np.concatenate([p[key] for p in parts]) == full[key]).all()
        cuts = sorted(set(rng.integers(1, c.B, size=3).tolist()))
        bounds = [0] + cuts + [c.B]
        parts = [o.rows(k, a, b) for a, b in zip(bounds, bounds[1:])]
        blob = b"".join(np.concatenate([p[key] for p in parts]).tobytes()
                        for key in ("tokens", "pos", "doc", "mask"))
        want = b"".join(full[key].tobytes() for key in ("tokens", "pos", "doc", "mask"))
        assert hashlib.sha256(blob).digest() == hashlib.sha256(want).digest()
        assert (full["row_learned"] == full["mask"].sum(1)).all()


def test_rows_follow_stream_and_rank_order():
    c = make_preset("c3s")
    o = oracle.Oracle(c)
    q, cum, _ = o.quota()
    firsts = [o.window_first(j) for j in range(c.n_streams)]
    pieces = [o.pieces(j) for j in range(c.n_streams)]
    for k in (0, 1, o.valid_steps - 1):
        r = o.rows(k)
        i = 0
        for j in range(c.n_streams):
            for x in range(int(q[k, j])):
                rank = int(cum[k, j]) + x
                p0 = int(firsts[j][rank])
                d, off, _ = (a[p0] for a in pieces[j])
                assert r["doc"][i, 0] == d
                assert r["tokens"][i, 0] == c.tokens[c.doc_offsets[d] + off]
                i += 1
        assert i == c.B


def test_exhaustion_horizon_and_drain():
    lengths = [30] * 10  # T = 32: every document is its own window
    c = corpus_from_lengths(lengths, T=32, B=4, max_steps=5)
    o = oracle.Oracle(c)
    assert o.n_windows(0) == 10
    assert o.valid_steps == 2         # step 2 would need windows 8..11
    with pytest.raises(oracle.OracleError) as e:
        o.rows(2)
    assert e.value.code == oracle.EXHAUSTED
    with pytest.raises(oracle.OracleError) as e:
        o.rows(5)
    assert e.value.code == oracle.HORIZON
    od = oracle.Oracle(c, drain=True)
    assert od.valid_steps == 3
    r = od.rows(2)
    assert (r["row_learned"] == [30, 30, 0, 0]).all()
    assert (r["doc"][2:] == -1).all() and (r["tokens"][2:] == c.pad_id).all()
    with pytest.raises(oracle.OracleError) as e:
        od.rows(3)
    assert e.value.code == oracle.EXHAUSTED


def test_bad_inputs_are_rejected():
    c = corpus_from_lengths([3, 4, 5], T=16, B=1, max_steps=1)
    c.doc_offsets = np.asarray([0, 3, 2, 12], np.int64)  # decreasing
    with pytest.raises(oracle.OracleError) as e:
        oracle.Oracle(c)
    assert e.value.code == oracle.BAD_INPUT
    c = corpus_from_lengths([3, 4, 5], T=16, B=1, max_steps=1)
    c.doc_offsets = np.asarray([0, 3, 7, 13], np.int64)  # past the tokens
    with pytest.raises(oracle.OracleError) as e:
        oracle.Oracle(c)
    assert e.value.code == oracle.BAD_INPUT
    c = corpus_from_lengths([3, 4, 5], T=16, B=1, max_steps=1, source_weight=[0])
    with pytest.raises(oracle.OracleError) as e:
        oracle.Oracle(c)
    assert e.value.code == oracle.INVALID_ARG


def test_order_digest():
    c = make_preset("c1")
    d0 = oracle.Oracle(c).digest
    assert oracle.Oracle(c).digest == d0
    assert oracle.Oracle(c, seed=1).digest != d0
    assert oracle.Oracle(c, max_steps=9).digest != d0
    c2 = make_preset("c1")
    c2.source_weight = np.asarray([6, 4], np.uint32)
    assert oracle.Oracle(c2).digest != d0


# ---- the row fingerprint's key layout, recovered key by key ------------------
# fp = mix(sum_t mix(key_t)) with key_t = a_t ^ ((b_t | t << 40) * golden),
# a_t = (u32 token << 32) | u32 doc and b_t = (mask << 32) | u32 pos.  Un-mixing
# a one-position row gives its key; in a two-position row whose first position
# is all zeros (key 0, term mix(0) = the first published SplitMix64 output)
# the second key follows the same way.  The expected keys are special cases
# worked out by hand: with b = 0 and t = 0 the key is a itself, and a product
# of the golden constant with a power of two is a shift of its hex digits.
# A swapped field, a shift of 32 instead of 40, an OR for the XOR or a missing
# multiply each gives another key.
SPLITMIX0 = 0xE220A8397B1DCDAF


def _one_pos(tok, pos, doc, mask):
    return dict(tokens=np.asarray([tok], np.int32), pos=np.asarray([pos], np.int32),
                doc=np.asarray([doc], np.int32), mask=np.asarray([mask], np.uint8))


def _key_t0(tok, pos, doc, mask):
    return _unmix(_unmix(_fp(_one_pos(tok, pos, doc, mask))))


def _key_t1(tok, pos, doc, mask):
    r = dict(tokens=np.asarray([0, tok], np.int32), pos=np.asarray([0, pos], np.int32),
             doc=np.asarray([0, doc], np.int32), mask=np.asarray([0, mask], np.uint8))
    return _unmix((_unmix(_fp(r)) - SPLITMIX0) & M64)


@pytest.mark.parametrize("tok,pos,doc,mask,key", [
    # b = 0, t = 0: the key is (token << 32) | doc
    (0x12345678, 0, 0x0BADF00D, 0, 0x123456780BADF00D),
    (-1, 0, -2, 0, 0xFFFFFFFFFFFFFFFE),
    (0, 0, -1, 0, 0x00000000FFFFFFFF),
    # a = 0: pos 1 -> golden; pos 2 -> 2 * golden; mask 1 -> golden << 32
    (0, 1, 0, 0, 0x9E3779B97F4A7C15),
    (0, 2, 0, 0, 0x3C6EF372FE94F82A),
    (0, 0, 0, 1, 0x7F4A7C1500000000),
    # both halves: (tok << 32 | doc) ^ golden
    (7, 1, 3, 0, 0x9E3779BE7F4A7C16),
])
def test_row_fingerprint_key_at_position_0(tok, pos, doc, mask, key):
    assert _key_t0(tok, pos, doc, mask) == key


@pytest.mark.parametrize("tok,pos,doc,mask,key", [
    # t = 1 adds 1 << 40 to b: golden << 40
    (0, 0, 0, 0, 0x4A7C150000000000),
    (7, 0, 3, 0, 0x4A7C150700000003),
    # (1 << 40 | 1) * golden = golden + golden << 40
    (0, 1, 0, 0, 0xE8B38EB97F4A7C15),
    # (1 << 40 | 1 << 32) * golden = golden << 40 + golden << 32
    (0, 0, 0, 1, 0xC9C6911500000000),
])
def test_row_fingerprint_key_at_position_1(tok, pos, doc, mask, key):
    assert _key_t1(tok, pos, doc, mask) == key


# ---- the order digest, item by item ------------------------------------------
# digest = mix(sum ^ count), sum = sum_i mix(item_i ^ mix(i)) over the items in
# their order: the recipe's scalars, each source's weight and held-out rate,
# each stream's document range, source and weight, the schedule, every valid
# update's quota row, and then, per stream, the first piece (doc << 32 | offset)
# of every window the valid updates read, in read order.  The items are taken
# here from the oracle's read-outs, each pinned on its own (quota tables, the
# packed pieces and windows, the read order); this checks that the digest
# covers exactly them.
def _digest_items(o, c, *, seed, G=0, bucket=0, drain=False, heldout_only=False,
                  shuffle_rows=False, wrap=False, schedule=None):
    v = o.valid_steps
    flags = (1 if drain else 0) | (2 if heldout_only else 0) | (4 if shuffle_rows else 0) | \
        (8 if wrap else 0)
    items = [c.T, c.B, c.max_steps, v, flags, c.pad_id & 0xFFFFFFFF, seed, c.hash_key,
             c.n_sources, c.n_streams, G, bucket]
    for s in range(c.n_sources):
        items += [int(c.source_weight[s]), int(c.source_heldout_bp[s])]
    for j in range(c.n_streams):
        items += [int(c.stream_doc_begin[j]), int(c.stream_doc_begin[j + 1]),
                  int(c.stream_source[j]), int(c.stream_weight[j])]
    if schedule:
        items.append(len(schedule))
        for p in schedule:
            items += [p["begin"], p["B"], *p["source_weight"], *p["stream_weight"]]
    q, cum, _ = o.quota()
    for k in range(v):
        items += [int(x) & M64 for x in q[k]]
    for j in range(c.n_streams):
        W = o.n_windows(j)
        used = min(int(cum[v, j]), W)
        doc, off, _ = o.pieces(j)
        first = o.window_first(j)
        for r in range(used):
            w = oracle.window_of_rank(seed, j, G, W, r)
            p = int(first[w])
            items.append((int(doc[p]) << 32) | int(off[p]))
    return items


def _fold_items(items):
    acc = 0
    for i, x in enumerate(items):
        acc = (acc + oracle.splitmix64((x & M64) ^ oracle.splitmix64(i))) & M64
    return acc ^ len(items)


@pytest.mark.parametrize("kw", [
    dict(),
    dict(window_segment=3, shuffle_rows=True),
    dict(drain=True, max_steps=40),
    dict(heldout_only=True),
    dict(wrap=True, len_bucket=64),
])
def test_order_digest_covers_exactly_its_items(kw):
    c = make_preset("c1")
    if "max_steps" in kw:
        c.max_steps = kw.pop("max_steps")
    o = oracle.Oracle(c, **kw)
    assert o.valid_steps > 0
    items = _digest_items(o, c, seed=c.seed, G=kw.get("window_segment", 0),
                          bucket=kw.get("len_bucket", 0), drain=kw.get("drain", False),
                          heldout_only=kw.get("heldout_only", False),
                          shuffle_rows=kw.get("shuffle_rows", False), wrap=kw.get("wrap", False))
    assert _unmix(o.digest) == _fold_items(items)


def test_order_digest_covers_a_schedule():
    c = corpus_from_lengths([5, 9, 3, 12, 7, 2, 8, 4] * 6, T=16, B=4, max_steps=6,
                            stream_docs=[16, 16, 16], stream_source=[0, 0, 1],
                            source_weight=[2, 1], stream_weight=[1, 1, 1])
    sched = [dict(begin=0, B=4, source_weight=[2, 1], stream_weight=[1, 1, 1]),
             dict(begin=3, B=3, source_weight=[1, 1], stream_weight=[1, 2, 1])]
    o = oracle.Oracle(c, schedule=sched)
    assert o.valid_steps > 3
    items = _digest_items(o, c, seed=c.seed, schedule=sched)
    assert _unmix(o.digest) == _fold_items(items)
