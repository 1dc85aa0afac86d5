"""The five workloads at full size, in the launch size the benchmark times
(its auto_launch updates per ns_pack_step launch -- at most 2^30 positions:
500 for the 512 x 4096 rows, 200 for 256 x 8192, 512 for 64 x 32768, the
whole horizon for the small-batch ones -- all rows of the global batch).

Every update of every workload is compared with the oracle on its row
fingerprints, learned counts, batch fingerprint and update learned count;
updates at launch boundaries and a few more are compared element by element.
Whole-pass properties (valid horizon, order digest, quota tables, exactly-once
coverage of a full long-context pass) are checked at any size.  Every update
of the elastic-determinism workload is also assembled in R = 8, 16, 32 and 64
row slices and compared byte for byte with the one-launch batch ("Zephon:
deterministic data loading": the SHA-256 of every global batch matches byte
for byte at any GPU count).
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import oracle
from _gpu import FIELDS, assert_rows_equal, batch_sha256, oracle_for, packer_for, to_host
from corpus import make_preset
from deterministic_packed_assembly_gb300 import as_u64

pytestmark = pytest.mark.gpu



def _launch(c):
    import bench
    return bench.auto_launch(c.max_steps, c.B, c.T)

_cache = {}


def _setup(name):
    if name not in _cache:
        c = make_preset(name)
        _cache[name] = (c, packer_for(c), oracle_for(c))
    return _cache[name]


def _one(out, q):
    """Update q of a launch's outputs, copied to the host alone."""
    return {f: v[0] for f, v in to_host({f: x[q:q + 1] for f, x in out.items()}).items()}


def _sampled(pk, o, steps, L):
    valid = o.valid_steps
    for k in steps:
        s0 = (k // L) * L
        n = min(L, valid - s0)
        out = pk.step(s0, n_steps=n)
        assert_rows_equal(_one(out, k - s0), o.rows(k), f"update {k}")
        del out
        assert pk.batch_fp(pk.step(k)["row_fp"][0]) == oracle.batch_fp(o.rows(k)["row_fp"])


def _tables(pk, o, c):
    assert pk.valid_steps == o.valid_steps
    assert pk.order_digest == o.digest
    q, cum = pk.quota_table()
    oq, ocum, _ = o.quota()
    assert (q == oq).all() and (cum == ocum).all()
    w, complete = pk.stream_windows()
    for j in range(c.n_streams):
        if complete[j]:
            assert w[j] == o.n_windows(j)
        else:
            assert ocum[-1, j] < w[j] <= o.n_windows(j)


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_full_size_sampled_updates(name):
    c, pk, o = _setup(name)
    # one init pass: neither the held-out hash's speculated bound nor the
    # shuffle of only the estimated prefix falls short on these workloads
    assert pk.info["init_passes"] == 1
    _tables(pk, o, c)
    v = o.valid_steps
    assert v > 0
    L = _launch(c)
    steps = sorted({0, 1, L - 1, L, v // 2, v - 2, v - 1} & set(range(v)))
    _sampled(pk, o, steps, L)
    pk.check()


def test_full_size_mixture_within_two_windows():
    c, pk, o = _setup("c3")
    # the held-out hash's speculated bound held for every stream
    assert pk.info["init_passes"] == 1
    q, _ = pk.quota_table()
    ss = c.stream_source.astype(np.int64)
    src = np.zeros((q.shape[0], c.n_sources), np.int64)
    for j in range(c.n_streams):
        src[:, ss[j]] += q[:, j]
    w = c.source_weight.astype(np.float64)
    share = c.B * w / w.sum()
    assert (np.abs(src - share[None, :]) <= 1).all()
    assert (src.sum(1) == c.B).all()


def _oracle_summaries(o, steps, full_rows=()):
    """Per update: the oracle's row fingerprints, row learned counts, batch
    fingerprint and update learned count, plus the whole rows of the updates
    in ``full_rows``.  The oracle's calls release the GIL and only read its
    built state, so updates are assembled on a few host threads; only the
    summaries are kept."""
    full_rows = set(full_rows)

    def one(k):
        r = o.rows(k)
        s = dict(row_fp=r["row_fp"], row_learned=r["row_learned"],
                 batch_fp=oracle.batch_fp(r["row_fp"]),
                 learned=int(r["row_learned"].astype(np.int64).sum()))
        if k in full_rows:
            s["rows"] = r
        return k, s

    with ThreadPoolExecutor(8) as ex:
        return dict(ex.map(one, steps))


def _boundary_updates(v, L):
    """Updates on both sides of the first launch boundaries and of the last."""
    ks = {0, 1, v // 2, v - 1}
    for s0 in list(range(L, v, L))[:3] + list(range(L, v, L))[-1:]:
        ks |= {s0 - 1, s0}
    return sorted(k for k in ks if 0 <= k < v)


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_full_size_every_update(name):
    # the whole horizon (c5: the drained full pass) in the benchmark's
    # launches; every update's row fingerprints, learned counts and batch
    # fingerprint equal the oracle's, and the updates at launch boundaries
    # equal it element by element
    c, pk, o = _setup(name)
    v = o.valid_steps
    L = _launch(c)
    full = _boundary_updates(v, L)
    want = _oracle_summaries(o, range(v), full)
    seen = 0
    for s0 in range(0, v, L):
        n = min(L, v - s0)
        out = pk.step(s0, n_steps=n)
        bfp = as_u64(pk.batch_fp_many(out["row_fp"]))
        upd = pk.step_learned(out["row_learned"]).cpu().numpy()
        got_fp = as_u64(out["row_fp"])
        got_l = out["row_learned"].cpu().numpy()
        for q in range(n):
            k = s0 + q
            w = want[k]
            assert (got_fp[q] == w["row_fp"]).all(), f"{name} update {k}: row_fp"
            assert (got_l[q] == w["row_learned"]).all(), f"{name} update {k}: row_learned"
            assert bfp[q] == w["batch_fp"], f"{name} update {k}: batch fingerprint"
            assert upd[q] == w["learned"], f"{name} update {k}: learned positions"
            if "rows" in w:
                assert_rows_equal(_one(out, q), w["rows"], f"{name} update {k}")
            seen += 1
        del out
    assert seen == v
    pk.check()


def test_full_size_elastic_slices_every_update():
    # every update of the elastic-determinism workload assembled once whole
    # and again as R = 8, 16, 32 and 64 independent row-slice launches into
    # poisoned buffers: all seven outputs byte-identical on the device, row
    # fingerprints equal to the oracle's, and the host SHA-256 of the four
    # [B, T] fields equal for every R on a sample of updates
    import torch
    c, pk, o = _setup("c4")
    v = o.valid_steps
    assert v == c.max_steps
    sha_sample = sorted({0, 1, v // 2, v - 1} | set(range(0, v, 25)))
    want = _oracle_summaries(o, range(v), sha_sample)
    Rs = (8, 16, 32, 64)
    bufs = {R: pk.empty_out(1) for R in Rs}
    for k in range(v):
        whole = pk.step(k)
        for R in Rs:
            b = bufs[R]
            for t in b.values():
                t.fill_(-3)
            for r in range(R):
                r0, r1 = r * c.B // R, (r + 1) * c.B // R
                pk.step(k, rows=(r0, r1), out={f: t[:, r0:r1] for f, t in b.items()})
            for f in b:
                assert torch.equal(b[f], whole[f]), (k, R, f)
        assert (as_u64(whole["row_fp"][0]) == want[k]["row_fp"]).all(), k
        if k in sha_sample:
            h = to_host(whole)
            one = {f: x[0] for f, x in h.items()}
            assert_rows_equal(one, want[k]["rows"], f"update {k}")
            sha = batch_sha256(one)
            for R in Rs:
                hb = {f: bufs[R][f][0].cpu().numpy() for f in FIELDS}
                assert batch_sha256(hb) == sha, (k, R)
    pk.check()


def test_full_size_long_context_full_pass_exactly_once():
    c, pk, o = _setup("c5")
    v = o.valid_steps
    real = 0
    learned = 0
    L = _launch(c)
    for s0 in range(0, v, L):
        n = min(L, v - s0)
        out = pk.step(s0, n_steps=n)
        real += int((out["doc"] >= 0).sum().item())
        learned += int(out["row_learned"].sum().item())
    # no held-out rate: every token of the corpus is assembled exactly once
    assert real == learned == c.n_tokens
    w, complete = pk.stream_windows()
    assert complete[0] and w[0] == o.n_windows(0)


@pytest.mark.parametrize("variant", ["heldout", "shuffled", "wrap", "schedule"])
def test_full_size_bench_variants(variant):
    # each packing option the benchmark times, on the benchmark's workload and
    # in its launch plan (32 updates per launch, never across a schedule piece)
    import torch
    import bench
    c = _setup("c3")[0]
    kw = bench.variant_kwargs(c, variant)
    pk, o = packer_for(c, **kw), oracle_for(c, **kw)
    assert pk.valid_steps == o.valid_steps > 0
    assert pk.order_digest == o.digest
    q, cum = pk.quota_table()
    oq, ocum, _ = o.quota()
    assert (q == oq).all() and (cum == ocum).all()
    w, complete = pk.stream_windows()
    for j in range(c.n_streams):
        if complete[j]:
            assert w[j] == o.n_windows(j)
        else:
            assert ocum[-1, j] <= w[j] <= o.n_windows(j)
    v = o.valid_steps
    plan = list(bench.launch_plan(pk, v, _launch(c)))
    want_steps = sorted({0, 1, v // 3, v // 2, v - 1} & set(range(v)))
    for s0, n, Bk in plan:
        hits = [k for k in want_steps if s0 <= k < s0 + n]
        if not hits:
            continue
        out = pk.step(s0, n_steps=n, rows=(0, Bk))
        for k in hits:
            assert_rows_equal(_one(out, k - s0), o.rows(k), f"update {k}")
        del out
    pk.close()
    del pk
    torch.cuda.empty_cache()


def test_full_size_host_corpus():
    # the 2M-document mixture handed over in page-locked host memory: copied
    # in groups of streams, each group hashed as it lands
    import torch
    from deterministic_packed_assembly_gb300 import Packer
    c, pk, o = _setup("c3")
    t = torch.from_numpy(c.tokens).pin_memory()
    off = torch.from_numpy(c.doc_offsets).pin_memory()
    import bench
    hp = Packer(t, off, None, device="cuda:0", **bench.recipe_kwargs(c))
    assert hp.order_digest == pk.order_digest == o.digest
    assert hp.valid_steps == pk.valid_steps
    L = _launch(c)
    v = o.valid_steps
    _sampled(hp, o, sorted({0, L, v - 1}), L)
    hp.close()
    del hp, t, off
    torch.cuda.empty_cache()
