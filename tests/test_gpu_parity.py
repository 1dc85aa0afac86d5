"""Parity of the CUDA library with the CPU oracle, element by element.

Integer work: the bar is bit-exact (tolerance 0) on every output -- tokens,
position ids, document ids, loss masks, row fingerprints, learned counts --
and on the bookkeeping (valid updates, windows per stream, quota tables, the
order digest).  Sizes here span many tiles and ragged tails while the oracle
stays fast; the full-size workloads are in test_gpu_full.py.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu import assert_rows_equal, batch_sha256, compare_steps, oracle_for, packer_for, to_host
from _helpers import corpus_from_lengths
from corpus import make_preset

pytestmark = pytest.mark.gpu


def _check_tables(pk, o, c):
    assert pk.valid_steps == o.valid_steps
    assert pk.order_digest == o.digest, (hex(pk.order_digest), hex(o.digest))
    q, cum = pk.quota_table()
    oq, ocum, _ = o.quota()
    assert (q == oq).all() and (cum == ocum).all()
    w, complete = pk.stream_windows()
    for j in range(c.n_streams):
        if complete[j]:
            assert w[j] == o.n_windows(j), j
        else:
            # a stream cut at its reachable prefix holds at least the windows
            # the horizon reads (greedy packing: one more, still open)
            assert ocum[-1, j] <= w[j] <= o.n_windows(j), j


@pytest.mark.parametrize("name", ["c1", "c2s", "c3s", "c4s", "c5s"])
def test_preset_every_step(name):
    c = make_preset(name)
    pk, o = packer_for(c), oracle_for(c)
    _check_tables(pk, o, c)
    assert o.valid_steps > 0
    compare_steps(pk, o, range(o.valid_steps), launch=4)
    pk.check()


@pytest.mark.parametrize("name", ["c1", "c3s"])
def test_slice_invariance(name):
    c = make_preset(name)
    pk, o = packer_for(c), oracle_for(c)
    for k in (0, o.valid_steps - 1):
        full = to_host(pk.step(k))
        want = o.rows(k)
        assert_rows_equal({f: v[0] for f, v in full.items()}, want, f"step {k}")
        digest = batch_sha256({f: v[0] for f, v in full.items()})
        fp = pk.batch_fp(pk.step(k)["row_fp"][0])
        assert fp == oracle.batch_fp(want["row_fp"])
        R = 1
        while R <= c.B:
            parts = [to_host(pk.step(k, rows=(r * c.B // R, (r + 1) * c.B // R))) for r in range(R)]
            cat = {f: np.concatenate([p[f][0] for p in parts]) for f in parts[0]}
            assert_rows_equal(cat, want, f"step {k} in {R} slices")
            assert batch_sha256(cat) == digest
            R *= 2


def test_multi_step_launch_equals_single_steps():
    c = make_preset("c4s")
    pk = packer_for(c)
    n = min(8, pk.valid_steps)
    many = to_host(pk.step(0, n_steps=n))
    for k in range(n):
        one = to_host(pk.step(k))
        assert_rows_equal({f: v[0] for f, v in one.items()}, {f: v[k] for f, v in many.items()},
                          f"step {k}")


def test_resume_in_a_fresh_context():
    c = make_preset("c3s")
    pk1 = packer_for(c)
    k = pk1.valid_steps // 2
    a = to_host(pk1.step(k))
    digest = pk1.order_digest
    pk1.close()
    pk2 = packer_for(c)
    assert pk2.order_digest == digest
    b = to_host(pk2.step(k))
    assert_rows_equal({f: v[0] for f, v in a.items()}, {f: v[0] for f, v in b.items()}, "resume")
    # a resume under another seed is another order: its digest differs
    assert packer_for(c, seed=1).order_digest != digest


def _random_case(rng):
    T = int(rng.choice([16, 32, 48, 64, 144]))
    J = int(rng.integers(1, 5))
    stream_docs = [int(rng.integers(0, 60)) for _ in range(J)]
    n = sum(stream_docs)
    lengths = []
    for _ in range(n):
        u = rng.random()
        if u < 0.06:
            lengths.append(0)
        elif u < 0.12:
            lengths.append(T * int(rng.integers(1, 3)))  # exactly T, 2T
        elif u < 0.75:
            lengths.append(int(rng.integers(1, T + 1)))
        else:
            lengths.append(int(rng.integers(T, 5 * T)))
    S = int(rng.integers(1, J + 1))
    stream_source = sorted(list(range(S)) + [int(x) for x in rng.integers(0, S, size=J - S)])
    B = int(rng.integers(1, 9))
    drain = bool(rng.integers(0, 2))
    bp = [int(rng.choice([0, 100, 3000, 10000])) for _ in range(S)]
    loss_start = None
    if rng.random() < 0.4:
        loss_start = [int(rng.integers(-3, max(L, 1) + 5)) for L in lengths]
    return corpus_from_lengths(
        lengths, T=T, B=B, max_steps=int(rng.integers(1, 40)), stream_docs=stream_docs,
        stream_source=stream_source, source_weight=[int(x) for x in rng.integers(1, 9, size=S)],
        stream_weight=[int(x) for x in rng.integers(1, 9, size=J)], heldout_bp=bp,
        loss_start=loss_start, seed=int(rng.integers(0, 2**63)),
        hash_key=int(rng.integers(0, 2**63)), drain=drain, pad_id=int(rng.integers(-5, 50000)))


@pytest.mark.parametrize("case", range(60))
def test_random_tiny_corpora(case):
    rng = np.random.default_rng(9000 + case)
    c = _random_case(rng)
    o = oracle_for(c)
    pk = packer_for(c)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=int(rng.integers(1, 5)))
    if o.valid_steps < c.max_steps:
        with pytest.raises(Exception) as e:
            pk.step(o.valid_steps)
        assert getattr(e.value, "code", None) == -4  # NS_ERR_EXHAUSTED
    pk.check()


def test_all_held_out_source_is_exhausted_at_once():
    c = corpus_from_lengths([30] * 8, T=32, B=2, max_steps=3, stream_docs=[4, 4],
                            heldout_bp=[10000, 0])
    pk, o = packer_for(c), oracle_for(c)
    assert pk.valid_steps == o.valid_steps == 0
    w, complete = pk.stream_windows()
    assert w[0] == 0 and complete[0]
    pkd, od = packer_for(c, drain=True), oracle_for(c, drain=True)
    assert pkd.valid_steps == od.valid_steps == 1
    compare_steps(pkd, od, [0])


def test_empty_streams_and_empty_documents():
    lengths = [0, 0, 5, 0, 40, 0, 17, 0]
    c = corpus_from_lengths(lengths, T=32, B=3, max_steps=6, stream_docs=[0, 4, 0, 4],
                            stream_source=[0, 0, 1, 1], drain=True)
    pk, o = packer_for(c), oracle_for(c)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps))


def test_documents_of_exactly_t_are_whole_windows():
    T = 64
    c = corpus_from_lengths([T] * 10 + [2 * T] * 3, T=T, B=4, max_steps=4)
    pk, o = packer_for(c), oracle_for(c)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps))
    r = to_host(pk.step(0))
    assert (r["row_learned"][0] == T).all()
    assert (r["pos"][0] == np.arange(T)[None, :]).all()


@pytest.mark.parametrize("wrap", [False, True])
def test_largest_window_length(wrap):
    # T at the library's limit (NS_MAX_T = 2^24): rows of 16 Mi positions,
    # documents longer than T (cut into a full chunk and a tail), a document
    # of the held-out hash 16 Mi tokens long, ragged ends everywhere
    T = 1 << 24
    lengths = [T + 37, 5, T - 3, 100, 3, T + 1]
    c = corpus_from_lengths(lengths, T=T, B=2, max_steps=3, heldout_bp=[1], drain=True)
    pk, o = packer_for(c, wrap=wrap), oracle_for(c, wrap=wrap)
    _check_tables(pk, o, c)
    assert o.valid_steps > 0
    compare_steps(pk, o, range(o.valid_steps))
    pk.check()
    pk.close()


def _medium_case(rng):
    """A mixture whose streams need hundreds to thousands of windows (the
    held-out hash speculates its bound for those past 256), documents
    log-normal around a random fraction of T (window fills from about 0.6 to
    nearly 1), some documents longer than T."""
    T = int(rng.choice([128, 256, 512]))
    J = int(rng.integers(2, 7))
    S = int(rng.integers(1, J + 1))
    stream_source = sorted(list(range(S)) + [int(x) for x in rng.integers(0, S, size=J - S)])
    B = int(rng.integers(24, 65))
    K = int(rng.integers(40, 121))
    med = T * float(rng.choice([0.05, 0.15, 0.3, 0.5, 0.9]))
    sigma = float(rng.uniform(0.4, 1.4))
    # documents per stream: enough for its share of K * B windows, with room
    sw = [int(x) for x in rng.integers(1, 9, size=S)]
    tw = [int(x) for x in rng.integers(1, 9, size=J)]
    mean_len = med * np.exp(sigma * sigma / 2)
    stream_docs = []
    for j in range(J):
        s = stream_source[j]
        share = sw[s] / sum(sw) * tw[j] / sum(tw[q] for q in range(J) if stream_source[q] == s)
        need = K * B * share * T / mean_len
        stream_docs.append(int(need * float(rng.uniform(1.3, 2.5))) + 50)
    n = sum(stream_docs)
    lengths = np.clip(np.rint(med * np.exp(sigma * rng.standard_normal(n))), 1, 4 * T).astype(int)
    bp = [int(rng.choice([50, 100, 500, 2000])) for _ in range(S)]
    loss_start = None
    if rng.random() < 0.3:
        loss_start = [int(rng.integers(0, L + 1)) for L in lengths]
    return corpus_from_lengths(
        lengths, T=T, B=B, max_steps=K, stream_docs=stream_docs, stream_source=stream_source,
        source_weight=sw, stream_weight=tw, heldout_bp=bp, loss_start=loss_start,
        seed=int(rng.integers(0, 2**63)), hash_key=int(rng.integers(0, 2**63)),
        drain=bool(rng.integers(0, 2)), tokens=rng.integers(0, 50000, size=int(lengths.sum())),
        pad_id=0)


@pytest.mark.parametrize("case", range(12))
def test_speculated_hash_bound_random_medium_corpora(case):
    # every update of mixtures large enough for the held-out hash to stop
    # at its speculated bound: tables and rows exactly the oracle's, whether
    # the bound held (one init pass) or a stream fell short (two)
    rng = np.random.default_rng(7000 + case)
    c = _medium_case(rng)
    kw = {}
    if rng.random() < 0.3:
        kw = dict(window_segment=int(rng.choice([4, 16])), shuffle_rows=True)
    o = oracle_for(c, **kw)
    # every third case from page-locked host memory, read in place
    if case % 3 == 1:
        _poison_cache(256 << 20)
        pk = _host_packer(c, True, **kw)
    else:
        pk = packer_for(c, **kw)
    assert pk.info["init_passes"] in (1, 2)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=int(rng.integers(4, 17)))
    pk.check()


def test_speculated_hash_bound_falls_short_and_init_runs_again():
    # the held-out hash stops at a bound speculated from the packing fill it
    # measures on a stream's first shuffled positions.  Here those hold
    # documents that fill a window poorly (33 of 64 tokens) and the later
    # ones documents that fill it fully (4 tokens): the measured fill (0.52)
    # leaves the stream short of the 4096 windows the horizon reads, and the
    # context is built again with the full bound -- same tables, same rows
    T, n_long, n_short, seed = 64, 2048, 40000, 3
    N = n_long + n_short
    lengths = np.zeros(N, np.int64)
    for p in range(N):
        lengths[oracle.feistel_pi(seed, 0, N, p)] = 33 if p < n_long else 4
    c = corpus_from_lengths(lengths, T=T, B=64, max_steps=64, heldout_bp=[1], seed=seed)
    pk, o = packer_for(c), oracle_for(c)
    assert pk.info["init_passes"] == 2
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=8)
    pk.check()
    # the same from page-locked host memory: both passes read it in place,
    # and both count in host_bytes
    _poison_cache()
    hp = _host_packer(c, True)
    assert hp.info["init_passes"] == 2
    assert hp.order_digest == pk.order_digest
    meta = (c.n_docs + 1) * 8
    assert hp.info["host_bytes"] - meta > c.n_tokens * 4 // 2
    compare_steps(hp, o, range(o.valid_steps), launch=8)
    hp.check()


@pytest.mark.parametrize("host", [False, True])
def test_hash_carries_a_stream_on_when_grabs_in_flight_keep_less_than_counted(host):
    # the held-out hash counts each grab in flight as keeping the stream's
    # expected fraction less 1/8 (here 10 % held out: 0.775) and takes no
    # more grabs once that count reaches the stream's need.  This stream's
    # shuffled positions [0, 40000) hold kept documents, the next 4000
    # held-out ones and the rest kept ones again, all of 16 tokens (four to a
    # window of 64).  The horizon's 10,000 windows hold exactly the first
    # 40000 and the need is one kept token more, so the grabs in flight at
    # the stop keep less than counted: the warp that decides the last of them
    # has to carry the stream through the held-out block on its own until a
    # kept document is decided.  Tables and rows are the oracle's
    T, L, seed, bp, key = 64, 16, 5, 1000, 0
    n_a, n_h, n_b = 40000, 4000, 16000
    N = n_a + n_h + n_b
    rng = np.random.default_rng(11)
    tokens = np.zeros((N, L), np.int32)
    for p in range(N):
        want = n_a <= p < n_a + n_h
        while True:
            t = rng.integers(0, 50000, size=L).astype(np.int32)
            if oracle.is_heldout(oracle.doc_hash(t, key), bp) == want:
                break
        tokens[oracle.feistel_pi(seed, 0, N, p)] = t
    c = corpus_from_lengths(np.full(N, L), T=T, B=100, max_steps=100, heldout_bp=[bp],
                            seed=seed, hash_key=key, tokens=tokens.ravel())
    o = oracle_for(c)
    assert int(o.heldout()[0].sum()) == n_h
    assert o.valid_steps == 100
    if host:
        _poison_cache()
        pk = _host_packer(c, True)
    else:
        pk = packer_for(c)
    assert pk.info["init_passes"] == 1
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=25)
    pk.check()


@pytest.mark.parametrize("host", [False, True])
def test_partial_shuffle_falls_short_and_init_runs_again(host):
    # a stream without a held-out rate is shuffled, on the first init pass,
    # only as far as the recipe's estimate of its windows' tokens over its
    # mean document length (a quarter and 1024 positions over).  Here its
    # first 20,000 shuffled positions hold 1-token documents and the other
    # 40,000 documents of 64 (one window each): the mean (43 tokens) puts
    # the 400 windows the horizon reads within about 1,800 positions, but
    # they take about 20,100.  The shortfall is caught after the cutoff and
    # the context is built again with every position -- same tables, same rows
    T, seed = 64, 9
    n_short, n_long = 20000, 40000
    N = n_short + n_long
    lengths = np.zeros(N, np.int64)
    for p in range(N):
        lengths[oracle.feistel_pi(seed, 0, N, p)] = 1 if p < n_short else 64
    c = corpus_from_lengths(lengths, T=T, B=8, max_steps=50, seed=seed)
    o = oracle_for(c)
    assert o.valid_steps == 50
    if host:
        _poison_cache()
        pk = _host_packer(c, True)
    else:
        pk = packer_for(c)
    assert pk.info["init_passes"] == 2
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=10)
    pk.check()


@pytest.mark.parametrize("name", ["c2s", "c3s"])
def test_step_learned_counts(name):
    # each update's learned positions: the sum of its rows' counts, in 64
    # bits, for whole batches and for row slices (whose counts add up)
    c = make_preset(name)
    pk, o = packer_for(c), oracle_for(c)
    n = o.valid_steps
    out = pk.step(0, n_steps=n)
    got = pk.step_learned(out["row_learned"]).cpu().numpy()
    want = np.asarray([int(o.rows(k)["row_learned"].astype(np.int64).sum()) for k in range(n)])
    assert (got == want).all()
    half = c.B // 2
    a = pk.step_learned(pk.step(0, n_steps=n, rows=(0, half))["row_learned"]).cpu().numpy()
    b = pk.step_learned(pk.step(0, n_steps=n, rows=(half, c.B))["row_learned"]).cpu().numpy()
    assert (a + b == want).all()


def test_horizon_and_row_range_errors():
    c = make_preset("c1")
    pk = packer_for(c)
    with pytest.raises(Exception) as e:
        pk.step(c.max_steps)
    assert e.value.code == -5  # NS_ERR_HORIZON
    with pytest.raises(Exception) as e:
        pk.step(c.max_steps - 1, n_steps=2)
    assert e.value.code == -5
    out = pk.empty_out(1, c.B)
    with pytest.raises(Exception) as e:
        pk.step(0, rows=(3, 3), out=out)
    assert e.value.code == -1
    with pytest.raises(Exception) as e:
        pk.step(0, rows=(0, c.B + 1), out=out)
    assert e.value.code == -1
    bad = dict(out)
    bad["tokens"] = torch.empty(c.B * c.T + 1, dtype=torch.int32, device="cuda:0")[1:]
    with pytest.raises(Exception) as e:
        pk.step(0, out=bad)
    assert e.value.code == -1


def test_misaligned_row_outputs_are_refused():
    # row fingerprints are stored as u64 and counts and lengths as int32: a
    # pointer not aligned for its type is refused on the host, before any
    # launch, by every call that takes one
    from deterministic_packed_assembly_gb300 import _lib as L
    c = make_preset("c1")
    pk = packer_for(c)
    out = pk.empty_out(1, c.B)
    raw = torch.zeros(c.B * 8 + 64, dtype=torch.uint8, device="cuda:0")
    a = raw.data_ptr()
    st = pk.stream.cuda_stream
    for field, off in (("row_fp", 4), ("row_learned", 2), ("row_len", 2)):
        bad = pk.prepare(out)
        setattr(bad, field, a + off)
        with pytest.raises(Exception) as e:
            pk.step(0, out=out, prepared=bad)
        assert e.value.code == -1, field
    for row_fp, dst in ((a + 4, a + 32), (a, a + 36)):
        with pytest.raises(Exception) as e:
            L.ns_pack_batch_fp(pk._ctx, row_fp, 1, c.B, dst, st)
        assert e.value.code == -1
    for learned, dst in ((a + 2, a + 32), (a, a + 36)):
        with pytest.raises(Exception) as e:
            L.ns_pack_step_learned(pk._ctx, learned, 1, c.B, dst, st)
        assert e.value.code == -1
    with pytest.raises(Exception) as e:
        L.ns_pack_fingerprint(pk._ctx, a + 4, c.B, st)
    assert e.value.code == -1
    torch.cuda.synchronize()
    assert int(raw.count_nonzero()) == 0  # nothing was written
    # the context is untouched: the same update, aligned, matches the oracle
    o = pk.step(0, out=out)
    torch.cuda.synchronize()
    want = oracle_for(c).rows(0)
    assert (o["row_fp"][0].cpu().numpy().view(np.uint64) == want["row_fp"]).all()
    pk.check()


def test_malformed_offsets_are_reported():
    c = corpus_from_lengths([3, 4, 5, 6], T=16, B=1, max_steps=2)
    c.doc_offsets = np.asarray([0, 3, 2, 12, 18], np.int64)
    with pytest.raises(Exception) as e:
        packer_for(c)
    assert e.value.code == -6  # NS_ERR_BAD_INPUT
    c.doc_offsets = np.asarray([0, 3, 7, 12, 19], np.int64)  # past the last token
    with pytest.raises(Exception) as e:
        packer_for(c)
    assert e.value.code == -6


def test_batch_fingerprints_many():
    c = make_preset("c1")
    pk, o = packer_for(c), oracle_for(c)
    out = pk.step(0, n_steps=o.valid_steps)
    fps = pk.batch_fp_many(out["row_fp"]).cpu().numpy().view(np.uint64)
    for k in range(o.valid_steps):
        assert fps[k] == oracle.batch_fp(o.rows(k)["row_fp"])


@pytest.mark.parametrize("S,strata", [(40, 2), (2, 40), (33, 1), (1, 33), (100, 1), (2, 100),
                                      (513, 1), (3, 300)])
def test_quota_tables_beyond_one_warp(S, strata):
    # more than 32 sources, or more than 32 strata in a source, take the
    # block-level quota kernels instead of the single-warp one; more than 64
    # children rank their shortfalls by a bitonic sort
    J = S * strata
    rng = np.random.default_rng(S * 100 + strata)
    lengths = [int(x) for x in rng.integers(1, 200, size=J * 6)]
    c = corpus_from_lengths(lengths, T=256, B=97, max_steps=7, stream_docs=[6] * J,
                            stream_source=[s for s in range(S) for _ in range(strata)],
                            source_weight=[int(x) for x in rng.integers(1, 1000, size=S)],
                            stream_weight=[int(x) for x in rng.integers(1, 1000, size=J)],
                            drain=True)
    pk, o = packer_for(c), oracle_for(c)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=3)


def test_largest_stream_count():
    # the most streams a recipe may have (1024 sources x 64 strata): the
    # cutoff's, row table's and digest's last blocks scan every stream, the
    # hash looks at streams 32 at a time, the quotas rank 1024 sources by a
    # bitonic sort; half the sources hold documents out
    S, strata = 1024, 64
    J = S * strata
    rng = np.random.default_rng(65536)
    lengths = rng.integers(1, 41, size=8 * J)
    c = corpus_from_lengths(lengths, T=64, B=4096, max_steps=4, stream_docs=[8] * J,
                            stream_source=[s for s in range(S) for _ in range(strata)],
                            source_weight=[int(x) for x in rng.integers(500, 1000, size=S)],
                            stream_weight=[int(x) for x in rng.integers(500, 1000, size=J)],
                            heldout_bp=[3000 * (s % 2) for s in range(S)], drain=True,
                            tokens=rng.integers(0, 32000, size=int(lengths.sum())))
    pk, o = packer_for(c), oracle_for(c)
    _check_tables(pk, o, c)
    assert o.valid_steps == 4
    compare_steps(pk, o, range(o.valid_steps), launch=2)


@pytest.mark.parametrize("max_steps", [2, 6, 40])
def test_both_held_out_sweeps(max_steps):
    # a short horizon stops hashing each stream once its kept tokens cover
    # its windows; a horizon past the data hashes all of it
    c = make_preset("c3s", max_steps=max_steps)
    pk, o = packer_for(c), oracle_for(c)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=2)


@pytest.mark.parametrize("name", ["c1", "c3s", "c5s"])
def test_validation_stream(name):
    # the held-out documents of every stream, packed and assembled the same way
    c = make_preset(name)
    if int(c.source_heldout_bp.max()) == 0:
        c.source_heldout_bp = np.full(c.n_sources, 700, np.uint16)
    pk = packer_for(c, heldout_only=True, drain=True)
    o = oracle_for(c, heldout_only=True, drain=True)
    _check_tables(pk, o, c)
    assert o.valid_steps > 0
    compare_steps(pk, o, range(o.valid_steps), launch=3)
    # and the training stream of the same recipe differs from it
    assert packer_for(c, drain=True).order_digest != pk.order_digest


@pytest.mark.parametrize("heldout", [False, True])
def test_heldout_rates_around_the_in_flight_estimate_bounds(heldout):
    # the held-out hash counts a grab in flight as keeping its stream's
    # expected fraction less 1/8, and nothing for a stream that keeps at most
    # 1/8: sources on both sides of that bound (kept fractions 1249, 1250 and
    # 1251 of 10000, of the training or of the validation stream) and far
    # from it, each a stream of 20,000 documents.  Tables and rows of every
    # update are the oracle's
    keep = [9999, 8751, 8750, 8749, 5000, 1251, 1250, 1249]
    bps = [k if heldout else 10000 - k for k in keep]
    rng = np.random.default_rng(99)
    n = 20000
    lengths = np.clip(np.rint(200 * np.exp(rng.standard_normal(n * len(bps)))), 1, 2048)
    c = corpus_from_lengths(lengths.astype(np.int64), T=512, B=8 * len(bps), max_steps=200,
                            stream_docs=[n] * len(bps), heldout_bp=bps, seed=17, hash_key=5,
                            drain=True,
                            tokens=rng.integers(0, 32000, size=int(lengths.sum())))
    kw = dict(heldout_only=heldout, drain=True)
    o = oracle_for(c, **kw)
    pk = packer_for(c, **kw)
    _check_tables(pk, o, c)
    assert o.valid_steps == 200
    compare_steps(pk, o, range(o.valid_steps), launch=16)
    pk.check()


@pytest.mark.parametrize("case", range(20))
def test_validation_stream_random_tiny_corpora(case):
    rng = np.random.default_rng(7000 + case)
    c = _random_case(rng)
    o = oracle_for(c, heldout_only=True)
    pk = packer_for(c, heldout_only=True)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=2)


@pytest.mark.parametrize("name,G,rows", [("c1", 1, False), ("c1", 3, True), ("c3s", 64, False),
                                         ("c3s", 7, True), ("c5s", 5, True), ("c4s", 0, True)])
def test_read_order_shuffles(name, G, rows):
    # windows read in a shuffled order within segments of G, rows of every
    # update shuffled: both are pure functions of the seed, so any slicing
    # still gives the oracle's bytes
    c = make_preset(name)
    pk = packer_for(c, window_segment=G, shuffle_rows=rows)
    o = oracle_for(c, window_segment=G, shuffle_rows=rows)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=3)
    k = o.valid_steps - 1
    half = c.B // 2
    compare_steps(pk, o, [k], rows=(half, c.B))


@pytest.mark.parametrize("case", range(20))
def test_read_order_random_tiny_corpora(case):
    rng = np.random.default_rng(8000 + case)
    c = _random_case(rng)
    G = int(rng.choice([0, 1, 2, 3, 9]))
    rows = bool(rng.integers(0, 2))
    o = oracle_for(c, window_segment=G, shuffle_rows=rows)
    pk = packer_for(c, window_segment=G, shuffle_rows=rows)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=2)


def _schedule_for(c, rng, n_pieces, K):
    begins = [0] + sorted(int(x) for x in rng.choice(np.arange(1, K), size=n_pieces - 1,
                                                       replace=False))
    return [dict(begin=b, B=int(rng.integers(1, c.B + 1)),
                 source_weight=[int(x) for x in rng.integers(1, 10**6, size=c.n_sources)],
                 stream_weight=[int(x) for x in rng.integers(1, 10**6, size=c.n_streams)])
            for b in begins]


@pytest.mark.parametrize("name,n_pieces,G,rows", [("c3s", 3, 0, False), ("c3s", 5, 4, True),
                                                  ("c1", 2, 0, True), ("c4s", 4, 0, False)])
def test_schedules(name, n_pieces, G, rows):
    # pieces of the horizon with their own rows per update and weights (a
    # mixture schedule and a batch-size ramp), with and without the read-order
    # shuffles
    c = make_preset(name)
    rng = np.random.default_rng(n_pieces * 10 + G)
    sched = _schedule_for(c, rng, n_pieces, c.max_steps)
    kw = dict(schedule=sched, window_segment=G, shuffle_rows=rows, drain=True)
    pk, o = packer_for(c, **kw), oracle_for(c, **kw)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=3)
    # a call may not ask for rows an update of it does not have
    small = [k for k in range(o.valid_steps) if pk.rows_of_step(k) < c.B]
    if small:
        with pytest.raises(Exception) as e:
            pk.step(small[0], rows=(0, pk.rows_of_step(small[0]) + 1))
        assert e.value.code == -1


@pytest.mark.parametrize("S,strata", [(40, 2), (2, 40), (130, 2), (2, 70)])
def test_schedules_beyond_one_warp(S, strata):
    J = S * strata
    rng = np.random.default_rng(S + strata)
    lengths = [int(x) for x in rng.integers(1, 200, size=J * 6)]
    c = corpus_from_lengths(lengths, T=256, B=97, max_steps=9, stream_docs=[6] * J,
                            stream_source=[s for s in range(S) for _ in range(strata)],
                            drain=True)
    sched = _schedule_for(c, rng, 3, 9)
    pk, o = packer_for(c, schedule=sched), oracle_for(c, schedule=sched)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=2)


@pytest.mark.parametrize("name,bucket,G,rows,heldout", [
    ("c1", 0, 0, False, False), ("c1", 16, 3, True, False), ("c3s", 256, 0, False, False),
    ("c3s", 0, 64, True, True), ("c4s", 48, 0, False, False), ("c5s", 1024, 5, True, False)])
def test_wrap_packing(name, bucket, G, rows, heldout):
    # windows of exactly T cut from each stream's concatenated kept tokens
    # (across document ends), with bucketed row lengths and every read-order
    # and validation option
    c = make_preset(name)
    kw = dict(wrap=True, len_bucket=bucket, window_segment=G, shuffle_rows=rows,
              heldout_only=heldout, drain=heldout)
    pk, o = packer_for(c, **kw), oracle_for(c, **kw)
    _check_tables(pk, o, c)
    assert pk.info["levels"] == 0
    assert o.valid_steps > 0
    compare_steps(pk, o, range(o.valid_steps), launch=3)
    k = o.valid_steps - 1
    compare_steps(pk, o, [k], rows=(c.B // 3, c.B))
    pk.check()


@pytest.mark.parametrize("case", range(30))
def test_wrap_random_tiny_corpora(case):
    rng = np.random.default_rng(6000 + case)
    c = _random_case(rng)
    kw = dict(wrap=True, len_bucket=int(rng.choice([0, 1, 16, 40, 1000])),
              window_segment=int(rng.choice([0, 0, 2, 5])), shuffle_rows=bool(rng.integers(0, 2)),
              heldout_only=bool(rng.random() < 0.25))
    o = oracle_for(c, **kw)
    pk = packer_for(c, **kw)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=int(rng.integers(1, 4)))
    if o.valid_steps < c.max_steps:
        with pytest.raises(Exception) as e:
            pk.step(o.valid_steps)
        assert getattr(e.value, "code", None) == -4  # NS_ERR_EXHAUSTED
    pk.check()


@pytest.mark.parametrize("wrap", [False, True])
def test_windows_of_many_short_documents(wrap):
    # windows of more than 32 pieces are read from the piece table instead of
    # the warp's registers; wrap windows there also start inside a document
    rng = np.random.default_rng(5 + wrap)
    lengths = [int(x) for x in rng.integers(1, 40, size=3000)]
    lengths[::97] = [int(x) for x in rng.integers(500, 3000, size=len(lengths[::97]))]
    loss_start = [int(rng.integers(0, L + 1)) for L in lengths]
    c = corpus_from_lengths(lengths, T=1024, B=6, max_steps=12, stream_docs=[1800, 1200],
                            stream_source=[0, 1], loss_start=loss_start, drain=True)
    kw = dict(wrap=wrap, len_bucket=128)
    pk, o = packer_for(c, **kw), oracle_for(c, **kw)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=2)


def test_bucketed_lengths_of_greedy_rows():
    c = make_preset("c3s")
    for bucket in (16, 100, c.T, 10 * c.T):
        pk, o = packer_for(c, len_bucket=bucket), oracle_for(c, len_bucket=bucket)
        _check_tables(pk, o, c)
        compare_steps(pk, o, [0, o.valid_steps - 1], launch=1)


def _host_packer(c, pinned=True, **kw):
    import torch
    from deterministic_packed_assembly_gb300 import Packer
    t = torch.from_numpy(np.ascontiguousarray(c.tokens))
    o = torch.from_numpy(np.ascontiguousarray(c.doc_offsets))
    ls = None if c.loss_start is None else torch.from_numpy(np.ascontiguousarray(c.loss_start))
    if pinned:
        t, o = t.pin_memory(), o.pin_memory()
        ls = None if ls is None else ls.pin_memory()
    args = dict(stream_doc_begin=c.stream_doc_begin, stream_source=c.stream_source,
                source_weight=c.source_weight, stream_weight=c.stream_weight,
                source_heldout_bp=c.source_heldout_bp, T=c.T, B=c.B, max_steps=c.max_steps,
                seed=c.seed, hash_key=c.hash_key, drain=c.drain, pad_id=c.pad_id)
    args.update(kw)
    return Packer(t, o, ls, device="cuda:0", **args)


def _poison_cache(nbytes=1 << 30):
    """Leave one block of nbytes filled with 0x7f in torch's caching allocator
    and nothing else, so that the next context's device memory (its copy of a
    host corpus included) starts as garbage rather than as a corpus an
    earlier test left behind."""
    import torch
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    torch.full((nbytes // 4,), 0x7F7F7F7F, dtype=torch.int32, device="cuda:0")
    torch.cuda.synchronize()


def _corpus_bytes(c):
    return c.n_tokens * 4 + (c.n_docs + 1) * 8 + (0 if c.loss_start is None else c.n_docs * 4)


@pytest.mark.parametrize("name,pinned,kw", [
    ("c1", True, {}), ("c1", False, {}), ("c1", True, {"heldout_only": True, "drain": True}),
    ("c2s", False, {}), ("c2s", True, {}), ("c3s", True, {}), ("c3s", False, {}),
    ("c3s", True, {"wrap": True}), ("c4s", True, {}), ("c5s", True, {}),
    ("c5s", True, {"heldout_only": True, "drain": True})])
def test_host_corpus(name, pinned, kw):
    # the corpus handed over in host memory gives the same context and rows:
    # page-locked tokens are read in place (the hash and the prefix copy write
    # what the horizon reaches into the library's device copy), other host
    # memory is copied whole, group by group as the hash goes
    c = make_preset(name)
    _poison_cache()
    pk = _host_packer(c, pinned, **kw)
    assert pk.host_corpus
    o = oracle_for(c, **kw)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=4)
    pk.check()
    host = pk.info["host_bytes"]
    meta = (c.n_docs + 1) * 8 + (0 if c.loss_start is None else c.n_docs * 4)
    if pinned:
        assert meta <= host <= _corpus_bytes(c)
    else:
        assert host == _corpus_bytes(c)
    ref = packer_for(c, **kw)
    assert pk.order_digest == ref.order_digest
    assert pk.info["table_bytes"] > ref.info["table_bytes"]  # it holds the corpus too
    assert ref.info["host_bytes"] == 0


def test_host_corpus_unaligned_page_locked_tokens_are_copied_whole():
    # page-locked tokens that do not start on a 16-byte boundary cannot be
    # read in place with 16-byte loads: the library copies them whole
    import torch
    from deterministic_packed_assembly_gb300 import Packer
    c = make_preset("c3s")
    buf = torch.empty(c.n_tokens + 1, dtype=torch.int32).pin_memory()
    buf[1:] = torch.from_numpy(c.tokens)
    t = buf[1:]
    assert t.data_ptr() % 16 != 0
    off = torch.from_numpy(c.doc_offsets).pin_memory()
    _poison_cache()
    pk = Packer(t, off, None, device="cuda:0", stream_doc_begin=c.stream_doc_begin,
                stream_source=c.stream_source, source_weight=c.source_weight,
                stream_weight=c.stream_weight, source_heldout_bp=c.source_heldout_bp, T=c.T,
                B=c.B, max_steps=c.max_steps, seed=c.seed, hash_key=c.hash_key)
    o = oracle_for(c)
    assert pk.info["host_bytes"] == _corpus_bytes(c)
    _check_tables(pk, o, c)
    compare_steps(pk, o, [0, 1, o.valid_steps - 1])
    pk.check()


@pytest.mark.parametrize("name", ["c3m", "c4s"])
def test_host_corpus_reads_only_the_reachable_prefix(name):
    # a horizon of two updates reaches a small part of the corpus: only its
    # documents cross the host link (held-out hash for the 200,000-document
    # mixture -- its warps' documents in flight when a stream stops are read
    # too -- the prefix copy for c4s, whose sources hold nothing out), and
    # its rows are exact
    c = make_preset(name, max_steps=2)
    _poison_cache()
    pk = _host_packer(c, True)
    o = oracle_for(c)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps))
    meta = (c.n_docs + 1) * 8
    tokens_read = pk.info["host_bytes"] - meta
    used = sum(int((o.rows(k)["doc"] >= 0).sum()) for k in range(o.valid_steps)) * 4
    assert used <= tokens_read < 0.5 * c.n_tokens * 4, (used, tokens_read, c.n_tokens * 4)


@pytest.mark.parametrize("name,limit", [("c3m", 1.2), ("c3s", 1.5)])
def test_host_corpus_hashes_little_past_the_need(name, limit):
    # the held-out hash stops each stream a little past the kept tokens its
    # windows need: the speculated margin, and the grabs still in flight when
    # the need is met (counted before a warp takes another, so the warps that
    # pile onto the last streams do not each add one).  The tokens it reads
    # from host memory stay within a fixed factor of the raw tokens of the
    # prefixes the horizon's windows take
    c = make_preset(name)
    pk = _host_packer(c, True)
    o = oracle_for(c)
    _, cum, _ = o.quota()
    bp = np.asarray(c.source_heldout_bp, np.float64)
    need = 0.0
    for j in range(c.n_streams):
        rmax = int(cum[-1, j])
        if rmax == 0:
            continue
        _, _, ln = o.pieces(j)
        wf = o.window_first(j)
        kept = int(ln[:int(wf[min(rmax, len(wf) - 1)])].astype(np.int64).sum())
        need += kept / (1.0 - bp[c.stream_source[j]] / 1e4)
    read = pk.info["host_bytes"] - (c.n_docs + 1) * 8
    ratio = read / (4.0 * need)
    print(f"{name}: read {read} B, need {4.0 * need:.4g} B, ratio {ratio:.4f}")
    assert 0.97 <= ratio <= limit, ratio


def _raw_config(c, tok, off, alloc, free, **flags):
    """A config for the C ABI built by hand (device corpus), for the tests that
    drive the entry points below the Python wrapper."""
    import deterministic_packed_assembly_gb300._lib as L
    keep = [np.ascontiguousarray(c.stream_doc_begin, np.uint32),
            np.ascontiguousarray(c.stream_source, np.uint32),
            np.ascontiguousarray(c.source_weight, np.uint32),
            np.ascontiguousarray(c.stream_weight, np.uint32),
            np.ascontiguousarray(c.source_heldout_bp, np.uint16)]
    cfg = L.ns_pack_config()
    cfg.tokens, cfg.n_tokens = tok.data_ptr(), tok.numel()
    cfg.doc_offsets, cfg.n_docs = off.data_ptr(), off.numel() - 1
    cfg.loss_start = None
    cfg.n_sources, cfg.n_streams, cfg.T = keep[2].size, keep[1].size, c.T
    cfg.stream_doc_begin, cfg.stream_source = keep[0].ctypes.data, keep[1].ctypes.data
    cfg.source_weight, cfg.stream_weight = keep[2].ctypes.data, keep[3].ctypes.data
    cfg.source_heldout_bp = keep[4].ctypes.data
    cfg.seed, cfg.hash_key, cfg.B, cfg.max_steps = c.seed, c.hash_key, c.B, c.max_steps
    cfg.flags = flags.get("flags", 0)
    cfg.alloc, cfg.free = alloc, free
    return cfg, keep


@pytest.mark.parametrize("wrap", [False, True])
def test_allocation_failures_release_everything(wrap):
    # the allocator fails at its n-th call, for every n the init makes: each
    # init returns NS_ERR_OOM and gives back every block it was handed
    import torch
    import deterministic_packed_assembly_gb300._lib as L
    c = make_preset("c3s")
    dev = torch.device("cuda:0")
    tok = torch.from_numpy(c.tokens).to(dev)
    off = torch.from_numpy(c.doc_offsets).to(dev)
    live, state = {}, {"calls": 0, "fail_at": None}

    def _alloc(nbytes, _user):
        state["calls"] += 1
        if state["fail_at"] is not None and state["calls"] == state["fail_at"]:
            return None
        p = torch.cuda.caching_allocator_alloc(int(nbytes), 0)
        live[p] = nbytes
        return p

    def _free(p, _user):
        assert p in live, "freed a block the allocator never handed out"
        del live[p]
        torch.cuda.caching_allocator_delete(p)

    a_cb, f_cb = L.ns_alloc_fn(_alloc), L.ns_free_fn(_free)
    flags = L.NS_PACK_WRAP if wrap else 0
    cfg, keep = _raw_config(c, tok, off, a_cb, f_cb, flags=flags)
    ctx = L.ns_pack_init(cfg)           # a clean run counts the calls
    total = state["calls"]
    assert total >= 2 and live
    L.ns_pack_free(ctx)
    assert not live
    for n in range(1, total + 1):
        state.update(calls=0, fail_at=n)
        with pytest.raises(L.NsPackError) as e:
            L.ns_pack_init(cfg)
        assert e.value.code == L.NS_ERR_OOM, n
        assert not live, (n, len(live))
    torch.cuda.synchronize()


def test_outputs_stay_inside_their_buffers():
    # every array is written exactly where the call says: canaries on both
    # sides of each output are untouched, and what lies between is the oracle's
    import torch
    c = make_preset("c3s")
    pk, o = packer_for(c, wrap=False), oracle_for(c)
    dev = pk.device
    k, n, r0, r1 = 1, 2, 3, c.B - 2
    rows = r1 - r0
    pad = 64  # elements on each side (keeps 16-byte alignment for every dtype)
    spec = dict(tokens=(torch.int32, c.T), pos=(torch.int32, c.T), doc=(torch.int32, c.T),
                mask=(torch.uint8, c.T), row_fp=(torch.int64, 1), row_learned=(torch.int32, 1),
                row_len=(torch.int32, 1))
    bufs, out = {}, {}
    for key, (dt, w) in spec.items():
        m = n * rows * w
        b = torch.full((m + 2 * pad,), 0x5A, dtype=dt, device=dev)
        bufs[key] = (b, m)
        shape = (n, rows, c.T) if w > 1 else (n, rows)
        out[key] = b[pad:pad + m].view(*shape)
    pk.step(k, n_steps=n, rows=(r0, r1), out=out)
    torch.cuda.synchronize()
    for key, (b, m) in bufs.items():
        h = b.cpu()
        assert (h[:pad] == 0x5A).all() and (h[pad + m:] == 0x5A).all(), key
    got = to_host(out)
    for q in range(n):
        assert_rows_equal({f: v[q] for f, v in got.items()}, o.rows(k + q, r0, r1), f"step {k + q}")


@pytest.mark.parametrize("case", range(40))
def test_every_option_together_random_tiny_corpora(case):
    # drain, validation stream, segments, row shuffle, wrap, buckets and a
    # schedule drawn together on random small corpora
    rng = np.random.default_rng(4000 + case)
    c = _random_case(rng)
    kw = dict(heldout_only=bool(rng.random() < 0.25), window_segment=int(rng.choice([0, 1, 3, 8])),
              shuffle_rows=bool(rng.integers(0, 2)), wrap=bool(rng.integers(0, 2)),
              len_bucket=int(rng.choice([0, 16, 48])))
    if c.max_steps >= 3 and rng.random() < 0.6:
        kw["schedule"] = _schedule_for(c, rng, int(rng.integers(2, min(4, c.max_steps) + 1)),
                                       c.max_steps)
    o = oracle_for(c, **kw)
    # every third case hands the corpus over in page-locked host memory
    if case % 3 == 2:
        _poison_cache(64 << 20)
        pk = _host_packer(c, True, **kw)
    else:
        pk = packer_for(c, **kw)
    _check_tables(pk, o, c)
    compare_steps(pk, o, range(o.valid_steps), launch=int(rng.integers(1, 4)))
    pk.check()


def test_free_without_waiting_keeps_queued_updates_right():
    # The Packer builds its contexts with NS_PACK_ORDERED_FREE: close() hands
    # the tables back to the caching allocator without waiting for the
    # stream, and the next context, built at once on the same stream, takes
    # the same blocks.  The updates queued before the close still read the
    # first context's tables (the second one's kernels come after them).
    c = make_preset("c3s")
    o = oracle_for(c)
    pk = packer_for(c)
    n = min(6, o.valid_steps)
    outs = [pk.step(k) for k in range(n)]
    pk.close()
    pk2 = packer_for(c, seed=c.seed + 1)
    out2 = pk2.step(0)
    for k in range(n):
        assert_rows_equal({f: v[0] for f, v in to_host(outs[k]).items()}, o.rows(k),
                          f"update {k}")
    o2 = oracle_for(c, seed=c.seed + 1)
    assert_rows_equal({f: v[0] for f, v in to_host(out2).items()}, o2.rows(0), "second context")
    pk2.close()


def test_free_after_a_step_on_another_stream_waits_for_it():
    # a step on a stream other than the context's: close() waits for the
    # device before the tables go back
    c = make_preset("c3s")
    o = oracle_for(c)
    pk = packer_for(c)
    side = torch.cuda.Stream()
    n = min(6, o.valid_steps)
    out = pk.empty_out(n)
    torch.cuda.synchronize()
    pk.step(0, n_steps=n, out=out, stream=side)
    pk.close()
    pk2 = packer_for(c, seed=c.seed + 1)
    side.synchronize()
    got = to_host(out)
    for k in range(n):
        assert_rows_equal({f: v[k] for f, v in got.items()}, o.rows(k), f"update {k}")
    pk2.close()


def test_probe_loop_computes_the_hash_terms():
    # the register-only loop that sets the hash kernel's arithmetic ceiling
    # computes the held-out hash's per-token term: its sum over one block of
    # five terms a thread equals the oracle's SplitMix64 of the same keys
    import deterministic_packed_assembly_gb300 as nsp
    acc = torch.zeros(1, dtype=torch.int64, device="cuda:0")
    nsp.ns_pack_probe_hash_terms(1, 5, acc.data_ptr())
    torch.cuda.synchronize()
    M = (1 << 64) - 1
    want = 0
    for g in range(256):
        tok = (g * 2654435761) & 0xFFFFFFFF
        for t in range(5):
            want = (want + oracle.splitmix64((((g & 1023) + t) << 32) | (tok ^ t))) & M
    assert int(acc.item()) & M == want


@pytest.mark.parametrize("at", [0, 126, 127, 128, 129, 255, 40 * 128 - 1, 40 * 128, 69998])
def test_malformed_offsets_far_from_the_horizon_are_reported(at):
    # 70,000 documents of two tokens; one document's offsets decrease (at 0:
    # the first offset is negative), far from the one window the horizon
    # reads: only the whole-array check sees it, at run boundaries of its
    # warps (128 offsets) and at the array's end
    c = corpus_from_lengths([2] * 70000, T=16, B=1, max_steps=1)
    offs = c.doc_offsets.copy()
    if at == 0:
        offs[0] = -1
    else:
        offs[at] = offs[at + 1] + 1
    c.doc_offsets = offs
    with pytest.raises(Exception) as e:
        packer_for(c)
    assert e.value.code == -6  # NS_ERR_BAD_INPUT
