"""The five workloads at full size, in the launch configuration the benchmark
times (its auto_launch updates per ns_pack_step launch -- 128 for the three
large workloads, the whole horizon for the small-batch ones -- all rows of
the global batch).

Sampled updates are compared element by element with the oracle; whole-pass
properties (valid horizon, order digest, quota tables, exactly-once coverage
of a full long-context pass, learned counts of every SFT update) are checked
at any size.  The elastic-determinism workload is also assembled in R = 8, 16,
32 and 64 row slices ("Zephon: deterministic data loading": the SHA-256 of
every global batch matches byte for byte at any GPU count).
"""
import numpy as np
import pytest
import oracle
from _gpu import assert_rows_equal, batch_sha256, oracle_for, packer_for, to_host
from corpus import make_preset

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


def test_full_size_sft_learned_counts_every_update():
    c, pk, o = _setup("c2")
    v = o.valid_steps
    L = _launch(c)
    for s0 in range(0, v, L):
        n = min(L, v - s0)
        out = pk.step(s0, n_steps=n)
        got_l = out["row_learned"].cpu().numpy()
        got_fp = out["row_fp"].cpu().numpy().view(np.uint64)
        step_l = pk.step_learned(out["row_learned"]).cpu().numpy()
        for q in range(n):
            want = o.rows(s0 + q)
            assert (got_l[q] == want["row_learned"]).all(), s0 + q
            assert (got_fp[q] == want["row_fp"]).all(), s0 + q
            assert step_l[q] == int(want["row_learned"].astype(np.int64).sum()), s0 + q


def test_full_size_elastic_slices():
    c, pk, o = _setup("c4")
    for k in (0, o.valid_steps - 1):
        full = to_host(pk.step(k))
        want = o.rows(k)
        assert_rows_equal({f: v[0] for f, v in full.items()}, want, f"update {k}")
        sha = batch_sha256({f: v[0] for f, v in full.items()})
        for R in (8, 16, 32, 64):
            parts = [to_host(pk.step(k, rows=(r * c.B // R, (r + 1) * c.B // R)))
                     for r in range(R)]
            cat = {f: np.concatenate([p[f][0] for p in parts]) for f in parts[0]}
            assert batch_sha256(cat) == sha, (k, R)
            assert (cat["row_fp"] == want["row_fp"]).all()


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
