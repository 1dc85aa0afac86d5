"""Helpers for the GPU parity tests: run the library, compare with the oracle."""
import hashlib

import numpy as np
import torch

import oracle
from deterministic_packed_assembly_gb300 import Packer, as_u64

FIELDS = ("tokens", "pos", "doc", "mask")


def packer_for(corpus, **overrides) -> Packer:
    return Packer.from_corpus(corpus, device="cuda:0", **overrides)


def oracle_for(corpus, **overrides) -> oracle.Oracle:
    return oracle.Oracle(corpus, **overrides)


def to_host(out: dict) -> dict:
    torch.cuda.synchronize()
    h = {k: out[k].cpu().numpy() for k in FIELDS}
    h["row_fp"] = as_u64(out["row_fp"])
    h["row_learned"] = out["row_learned"].cpu().numpy()
    h["row_len"] = out["row_len"].cpu().numpy()
    return h


def assert_rows_equal(got: dict, want: dict, what: str) -> None:
    for k in FIELDS + ("row_fp", "row_learned", "row_len"):
        g, w = got[k], want[k]
        assert g.shape == w.shape, (what, k, g.shape, w.shape)
        if not np.array_equal(g, w):
            bad = np.argwhere(g != w)
            first = tuple(bad[0])
            raise AssertionError(f"{what}: {k} differs at {len(bad)} places, first {first}: "
                                 f"got {g[first]} want {w[first]}")


def compare_steps(pk: Packer, o: oracle.Oracle, steps, launch: int = 1, rows=None) -> None:
    """Assemble `steps` (consecutive runs batched `launch` at a time) and
    compare every element with the oracle."""
    steps = list(steps)
    i = 0
    while i < len(steps):
        s0 = steps[i]
        r0, r1 = (0, pk.rows_of_step(s0)) if rows is None else rows
        n = 1
        while (n < launch and i + n < len(steps) and steps[i + n] == s0 + n
               and pk.rows_of_step(s0 + n) == pk.rows_of_step(s0)):
            n += 1
        got = to_host(pk.step(s0, n_steps=n, rows=(r0, r1)))
        for q in range(n):
            want = o.rows(s0 + q, r0, r1)
            assert_rows_equal({k: v[q] for k, v in got.items()}, want,
                              f"step {s0 + q} rows [{r0},{r1})")
        i += n


def batch_sha256(rows: dict) -> bytes:
    h = hashlib.sha256()
    for k in FIELDS:
        h.update(np.ascontiguousarray(rows[k]).tobytes())
    return h.digest()
