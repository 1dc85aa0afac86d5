"""Multi-rank host logic of the benchmark, on CPU with the gloo backend.

Each rank assembles its own slice of rows of every update; the slices must
partition the global batch, and the timing reduction takes the maximum over
ranks.  The oracle shows that the rows each rank would produce concatenate to
the global batch.
"""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, B, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import bench
    d = bench.Dist()
    r0, r1 = bench.row_slice(rank, world, B)
    m = d.max(float(rank + 1) * 1.5)
    s = d.sum(float(r1 - r0))
    d.barrier()
    d.close()
    q.put((rank, r0, r1, m, s))


@pytest.mark.parametrize("world,B", [(2, 512), (3, 16), (4, 64)])
def test_ranks_partition_rows_and_take_the_max(world, B):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, world, port, B, q)) for r in range(world)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    cover = []
    for rank, r0, r1, m, s in res:
        cover.extend(range(r0, r1))
        assert m == world * 1.5
        assert s == B
    assert cover == list(range(B))


def test_rank_slices_concatenate_to_the_global_batch():
    import bench
    import oracle
    from corpus import make_preset
    c = make_preset("c1")
    o = oracle.Oracle(c)
    full = o.rows(3)
    for world in (2, 4, 8):
        parts = [o.rows(3, *bench.row_slice(r, world, c.B)) for r in range(world)]
        for k in full:
            assert np.array_equal(np.concatenate([p[k] for p in parts]), full[k])


def test_launch_plan_equal_launches_within_each_piece():
    # the benchmark's launches: the fewest that keep each within the most a
    # launch takes, equal in size within a schedule piece (the last one at
    # most as long as the others), never across a piece
    import bench

    class One:
        schedule = None

        @staticmethod
        def rows_of_step(k):
            return 64

    def sizes(plan_of, valid, L):
        return [m for _, m, _ in bench.launch_plan(plan_of, valid, L)]

    assert sizes(One, 574, bench.auto_launch(1024, 64, 32768)) == [287, 287]
    assert sizes(One, 1000, bench.auto_launch(1000, 512, 4096)) == [500, 500]
    assert sizes(One, 200, bench.auto_launch(200, 256, 8192)) == [200]
    assert sizes(One, 500, bench.auto_launch(500, 8, 4096)) == [500]
    for valid in range(1, 60):
        for L in range(1, 20):
            m = sizes(One, valid, L)
            assert sum(m) == valid and max(m) <= L and len(m) == -(-valid // L)
            # all equal but the last, which is no longer than the others
            assert len(set(m[:-1])) <= 1 and m[-1] <= m[0]

    class Pieces:
        schedule = [{"begin": 0, "B": 4}, {"begin": 7, "B": 8}]

        @staticmethod
        def rows_of_step(k):
            return 4 if k < 7 else 8

    plan = list(bench.launch_plan(Pieces, 20, 5))
    assert [(s, m) for s, m, _ in plan] == [(0, 4), (4, 3), (7, 5), (12, 5), (17, 3)]
    assert all(b == Pieces.rows_of_step(s) for s, _, b in plan)


def test_schedule_launch_plan_slices_cover_every_update():
    # the benchmark's launches never cross a schedule piece, and under any rank
    # count the ranks' slices of each launch concatenate to the global rows
    import bench
    import oracle
    from corpus import make_preset
    c = make_preset("c1")
    kw = bench.variant_kwargs(c, "schedule")

    class Plan:
        schedule = kw["schedule"]

        @staticmethod
        def rows_of_step(k):
            return [p["B"] for p in kw["schedule"] if p["begin"] <= k][-1]

    o = oracle.Oracle(c, **kw)
    v = o.valid_steps
    assert v > 0
    plan = list(bench.launch_plan(Plan, v, 3))
    assert [s for s, _, _ in plan] == sorted(s for s, _, _ in plan)
    assert sum(m for _, m, _ in plan) == v
    for s0, m, Bk in plan:
        assert all(Plan.rows_of_step(s0 + q) == Bk for q in range(m))
    for world in (2, 3):
        for s0, m, Bk in plan:
            for q in range(m):
                parts = [o.rows(s0 + q, *bench.row_slice(r, world, Bk)) for r in range(world)
                         if bench.row_slice(r, world, Bk)[1] > bench.row_slice(r, world, Bk)[0]]
                full = o.rows(s0 + q)
                for f in full:
                    assert np.array_equal(np.concatenate([p[f] for p in parts]), full[f])


class _Plan:
    """The piece of a Packer that bench.launch_plan reads."""

    def __init__(self, schedule, B):
        self.schedule, self.B = schedule, B

    def rows_of_step(self, k):
        if not self.schedule:
            return self.B
        return [p["B"] for p in self.schedule if p["begin"] <= k][-1]


def _collective_worker(rank, world, port, variant, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import torch
    import bench
    import oracle
    from corpus import make_preset
    c = make_preset("c1")
    kw = bench.variant_kwargs(c, variant)
    o = oracle.Oracle(c, **kw)
    v = o.valid_steps
    plan = list(bench.launch_plan(_Plan(kw.get("schedule"), c.B), v, 3))
    d = bench.Dist()
    # this rank's slice of every update, computed by the oracle: its row
    # fingerprints (padded to the largest slice) and its learned positions
    n_buf = -(-c.B // world)
    local = torch.zeros((v, n_buf), dtype=torch.int64)
    learned = torch.zeros(v, dtype=torch.int64)
    for s0, m, Bk in plan:
        r0, r1 = bench.row_slice(rank, world, Bk)
        for k in range(s0, s0 + m):
            if r1 > r0:
                rows = o.rows(k, r0, r1)
                local[k, :r1 - r0] = torch.from_numpy(rows["row_fp"].view(np.int64))
                learned[k] = int(rows["row_learned"].astype(np.int64).sum())
    bench.reduce_learned(d, learned)
    runs = bench.fold_runs(plan)
    got = bench.gather_batch_rows(d, local, runs, world)
    d.barrier()
    d.close()
    q.put((rank, learned.numpy(), [(f0, fm, g.numpy()) for (f0, fm, _), g in zip(runs, got)]))


@pytest.mark.parametrize("world,variant", [(2, "default"), (4, "default"), (3, "schedule")])
def test_row_split_collectives_rebuild_every_global_batch(world, variant):
    # the two collectives of a row split over ranks: each update's learned
    # positions summed over the ranks' slices, and the row fingerprints
    # gathered in row order, whose fold is the global batch fingerprint --
    # both equal to what one rank holding the whole batch gets
    import bench
    import oracle
    from corpus import make_preset
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_collective_worker, args=(r, world, port, variant, q))
          for r in range(world)]
    for p in ps:
        p.start()
    res = sorted((q.get(timeout=180) for _ in range(world)), key=lambda x: x[0])
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    c = make_preset("c1")
    o = oracle.Oracle(c, **bench.variant_kwargs(c, variant))
    v = o.valid_steps
    want = [o.rows(k) for k in range(v)]
    for rank, learned, runs in res:
        assert [int(x) for x in learned] == [int(w["row_learned"].astype(np.int64).sum())
                                             for w in want]
        covered = 0
        for f0, fm, rows in runs:
            for i in range(fm):
                k = f0 + i
                fp = rows[i].view(np.uint64)
                assert np.array_equal(fp, want[k]["row_fp"]), (rank, k)
                assert oracle.batch_fp(fp) == oracle.batch_fp(want[k]["row_fp"])
                covered += 1
        assert covered == v
