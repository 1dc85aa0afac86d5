"""The entry point that allocates no device memory: ns_pack_quota_noalloc.

It serves callers that cannot call cudaMalloc -- a trainer that gave all of
the GPU's memory to its own pool at start-up, a process held to a fixed
memory budget on a shared GPU, or a loop that cannot pay for the device
synchronisation cudaMalloc and cudaFree bring.  Its scratch is one static
device array shared by every call, so these tests check that two calls in a
row, through the C ABI, each give exactly the quota tables the allocating
path (ns_pack_init, read back with ns_pack_quota_table) builds for the same
recipe -- one recipe within a warp's reach and one that needs the scratch
table of per-update source windows -- and that a call returns without waiting
for the work already queued on its stream.  This file is named to run last.
"""
import numpy as np
import pytest
import torch

from _helpers import corpus_from_lengths
from corpus.synthetic import _preset_kwargs

pytestmark = pytest.mark.gpu


def _recipes():
    kw = _preset_kwargs("c3")  # 15 sources x 3 strata: the single-warp kernel
    mixture = dict(source_weight=kw["source_weight"], stream_source=kw["stream_source"],
                   stream_weight=kw["stream_weight"], B=512, max_steps=1000)
    rng = np.random.default_rng(77)  # 40 sources x 2 strata: needs the scratch table
    wide = dict(source_weight=[int(x) for x in rng.integers(1, 10**6, size=40)],
                stream_source=[s for s in range(40) for _ in range(2)],
                stream_weight=[int(x) for x in rng.integers(1, 10**6, size=80)],
                B=300, max_steps=400)
    # 130 sources x 1 stratum: the source level ranks its shortfalls by sorting
    many = dict(source_weight=[int(x) for x in rng.integers(1, 10**6, size=130)],
                stream_source=list(range(130)),
                stream_weight=[1] * 130, B=257, max_steps=300)
    return [("mixture", mixture), ("forty_sources", wide), ("many_sources", many)]


def _tables_by_init(r):
    """The allocating path: a context over a tiny corpus with the recipe."""
    from deterministic_packed_assembly_gb300 import Packer
    J = len(r["stream_source"])
    c = corpus_from_lengths([1] * J, T=16, B=r["B"], max_steps=r["max_steps"],
                            stream_docs=[1] * J, stream_source=r["stream_source"],
                            source_weight=r["source_weight"], stream_weight=r["stream_weight"])
    pk = Packer.from_corpus(c, device="cuda:0")
    q, cum = pk.quota_table()
    pk.close()
    return q, cum


def _tables_no_alloc(r, quota_dev, cum_dev):
    import deterministic_packed_assembly_gb300 as nsp
    nsp.ns_pack_quota_noalloc(r["source_weight"], r["stream_source"], r["stream_weight"],
                              r["B"], r["max_steps"], quota_dev.data_ptr(), cum_dev.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return quota_dev.cpu().numpy(), cum_dev.cpu().numpy()


def test_two_calls_in_a_row_match_the_allocating_path():
    recipes = _recipes()
    want = {name: _tables_by_init(r) for name, r in recipes}
    # two calls in a row per recipe, then the recipes interleaved, each into
    # buffers the caller owns (filled with garbage first)
    order = [recipes[0], recipes[0], recipes[1], recipes[1], recipes[2], recipes[2],
             recipes[0]]
    for name, r in order:
        K, J = r["max_steps"], len(r["stream_source"])
        q_dev = torch.full((K, J), -7, dtype=torch.int32, device="cuda:0")
        c_dev = torch.full((K + 1, J), -7, dtype=torch.int32, device="cuda:0")
        q, cum = _tables_no_alloc(r, q_dev, c_dev)
        wq, wc = want[name]
        assert np.array_equal(q, wq), name
        assert np.array_equal(cum, wc), name


def test_call_does_not_wait_on_its_stream():
    # a kernel that keeps the stream busy for about half a second is queued
    # first; the call must return long before it ends (the recipe travels in
    # kernel parameters, not in a copy from pageable memory that would wait
    # for the stream), and its tables must still be right once it has run.
    # 64 sources x 1000 strata: the upload takes nine launches.
    import time
    r = dict(source_weight=[1 + (s % 5) for s in range(64)],
             stream_source=[s for s in range(64) for _ in range(1000)],
             stream_weight=[1 + (j % 7) for j in range(64000)], B=4096, max_steps=4)
    K, J = r["max_steps"], len(r["stream_source"])
    q_dev = torch.full((K, J), -7, dtype=torch.int32, device="cuda:0")
    c_dev = torch.full((K + 1, J), -7, dtype=torch.int32, device="cuda:0")
    st = torch.cuda.current_stream()
    import deterministic_packed_assembly_gb300 as nsp
    torch.cuda.synchronize()
    torch.cuda._sleep(int(1e9))  # about 0.5 s at the SM clock
    t0 = time.perf_counter()
    nsp.ns_pack_quota_noalloc(r["source_weight"], r["stream_source"], r["stream_weight"],
                              r["B"], r["max_steps"], q_dev.data_ptr(), c_dev.data_ptr(),
                              st.cuda_stream)
    t_call = time.perf_counter() - t0
    busy = not st.query()
    torch.cuda.synchronize()
    t_all = time.perf_counter() - t0
    assert busy, "the queued kernel ended before the call returned"
    assert t_call < 0.5 * t_all, (t_call, t_all)
    q, cum = q_dev.cpu().numpy(), c_dev.cpu().numpy()
    wq, wc = _tables_by_init(r)
    assert np.array_equal(q, wq) and np.array_equal(cum, wc)


def test_recipe_beyond_the_scratch_is_rejected():
    import deterministic_packed_assembly_gb300 as nsp
    S = 1024  # 1024 sources x 2100 updates x 4 bytes does not fit in 8 MiB
    q_dev = torch.empty(1, dtype=torch.int32, device="cuda:0")
    with pytest.raises(nsp.NsPackError) as e:
        nsp.ns_pack_quota_noalloc([1] * S, list(range(S)), [1] * S, 8, 2100, q_dev.data_ptr(),
                                  q_dev.data_ptr())
    assert e.value.code == nsp.NS_ERR_INVALID_ARG
