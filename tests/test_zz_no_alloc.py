"""The entry point that allocates no device memory: ns_pack_quota_noalloc.

It serves callers that cannot call cudaMalloc -- a trainer that gave all of
the GPU's memory to its own pool at start-up, a process held to a fixed
memory budget on a shared GPU, or a loop that cannot pay for the device
synchronisation cudaMalloc and cudaFree bring.  Its scratch is one static
device array shared by every call, so these tests check that two calls in a
row, through the C ABI, each give exactly the quota tables the allocating
path (ns_pack_init, read back with ns_pack_quota_table) builds for the same
recipe -- one recipe within a warp's reach and one that needs the scratch
table of per-update source windows.  This file is named to run last.
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


def test_recipe_beyond_the_scratch_is_rejected():
    import deterministic_packed_assembly_gb300 as nsp
    S = 1024  # 1024 sources x 2100 updates x 4 bytes does not fit in 8 MiB
    q_dev = torch.empty(1, dtype=torch.int32, device="cuda:0")
    with pytest.raises(nsp.NsPackError) as e:
        nsp.ns_pack_quota_noalloc([1] * S, list(range(S)), [1] * S, 8, 2100, q_dev.data_ptr(),
                                  q_dev.data_ptr())
    assert e.value.code == nsp.NS_ERR_INVALID_ARG
