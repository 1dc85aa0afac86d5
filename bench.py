#!/usr/bin/env python3
"""Benchmark: packed tokens/s of deterministic packed assembly on GB300.

One bench step is one whole pass of the packing path over the workload: the
context build (held-out hash of every document, Feistel shuffle of every
stream, scans, piece expansion, next-window search, pointer jumping, window
numbering, two-level quotas, order digest) followed by the assembly of every
update of the horizon (row gather with position ids, document ids, loss
masks, row fingerprints, learned counts) and the batch fingerprint and
learned positions of every update.  Inputs are resident in HBM when the timed
region starts; outputs go to a reused device buffer of ``--launch`` updates.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c3]
    python bench.py --impl reference ...     # the CPU oracle on the same workload

Prints one JSON line (rank 0).  Under torchrun each rank assembles its own
slice of rows of every update (the same global batch, split by rows) with no
data-path collective; the timed region is bracketed by barriers and the
maximum over ranks is taken.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

WORKLOADS = {
    "c1": "2 sources x 5,000 docs, log-normal median 200 sigma 1.0 [1,8192], vocab 32,000, "
          "shares 7:3, 1 % held out, T=1024, B=16, 10 updates",
    "c2": "SFT packing: 200,000 prompt/completion examples (medians 64/128, sigma 1.0, "
          "<=4096), vocab 128,256, completion-only mask, T=4096, B=8, 500 updates",
    "c3": "15-source mixture x 3 strata (Dirichlet(1) shares, seed 1), 2,000,000 docs "
          "log-normal median 600 sigma 1.2 [1,65536], vocab 64,000, 1 % held out (5 % for "
          "source 15), T=4096, B=512, 1000 updates",
    "c3m": "a tenth of c3: 200,000 docs, same shape, T=4096, B=512, 96 updates",
    "c4": "4 equal sources x 2,000,000 docs log-normal median 400 sigma 1.0, vocab 50,257, "
          "T=8192, B=256, 200 updates",
    "c4m": "a tenth of c4: 4 x 200,000 docs, same shape, T=8192, B=256, 64 updates",
    "c5": "1 source of ~1e9 tokens, log-normal median 2048 sigma 1.5 [1,262144], vocab "
          "151,936, T=32768, B=64, long documents cut into T-chunks, full pass (drain)",
    "c5m": "a tenth of c5: 1 source of ~1e8 tokens, same shape, T=32768, B=64, full pass "
           "(drain)",
}
VARIANTS = {
    "default": "training stream, greedy packing cut at document ends, windows and rows in order",
    "heldout": "validation stream: the held-out documents of every stream, same shuffle, "
               "packing and quotas (drain)",
    "shuffled": "windows read in a keyed order within segments of 64, rows of every update "
                "shuffled",
    "wrap": "wrap packing: windows of exactly T across document ends, row lengths rounded "
            "up to buckets of 256",
    "schedule": "4-piece schedule: batch ramp B/4, B/2, 3B/4, B rows from updates 0, K/8, "
                "K/4, K/2, each piece with the recipe's weights scaled by draws in "
                "[0.8, 1.25) (seed 77)",
}
METRIC = "packed tokens/s"
L2_BYTES = 129e6
UNIT = "tokens/s"
PROFILES = os.path.join(ROOT, "profiles")
GATHER_SRC = os.path.join(ROOT, "deterministic_packed_assembly_gb300", "csrc", "gather.cu")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="c3", choices=sorted(WORKLOADS))
    ap.add_argument("--launch", type=int, default=0,
                    help="updates per ns_pack_step launch (0: equal launches of at most 2^30 positions "
                         "per launch, see auto_launch)")
    ap.add_argument("--slices", type=int, default=1,
                    help="split every launch into this many row-slice launches (the same "
                         "bytes per row; batch folds are skipped when > 1)")
    ap.add_argument("--variant", default="default", choices=sorted(VARIANTS),
                    help="packing options of the pass (validation stream, read-order "
                         "shuffles, wrap packing, schedule)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--also", default="c4",
                    help="comma-separated workloads also measured (no CPU baseline) and "
                         "reported under extra_configs; 'none' for none")
    return ap.parse_args()


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---- distributed plumbing ---------------------------------------------------
class Dist:
    def __init__(self):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def row_slice(rank: int, world: int, B: int) -> tuple[int, int]:
    """Rows of the global batch that rank `rank` of `world` assembles."""
    return rank * B // world, (rank + 1) * B // world


# ---- clocks -----------------------------------------------------------------
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
REJECT = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons; the
    samples taken between mark() and stop() describe the timed region (if it
    was too short to hold one, the last sample before it stands in, flagged
    ``nearest_before``)."""

    def __init__(self, gpu_id: str):
        self.f = tempfile.NamedTemporaryFile("w+", delete=False, suffix=".csv")
        self.offset = 0
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             + ",".join("clocks_event_reasons." + r for r in REASONS))
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
            return
        # sampling is live before the timed region starts
        t_end = time.time() + 5.0
        while time.time() < t_end and os.path.getsize(self.f.name) == 0:
            time.sleep(0.01)

    def mark(self) -> None:
        """The timed region starts: later samples are the region's."""
        if self.p is not None:
            self.offset = os.path.getsize(self.f.name)

    def stop(self) -> dict | None:
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        text = self.f.read()
        os.unlink(self.f.name)
        before, inside = text[:self.offset], text[self.offset:]
        rows = [ln.strip().split(", ") for ln in inside.splitlines() if ln.strip()]
        nearest = False
        if not rows:
            prev = [ln.strip().split(", ") for ln in before.splitlines() if ln.strip()]
            rows, nearest = prev[-1:], True
        sm, mx, seen = [], [], set()
        for r in rows:
            if len(r) < 4 + len(REASONS):
                continue
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except ValueError:
                continue
            for name, v in zip(REASONS, r[4:]):
                if v.strip().lower() == "active":
                    seen.add(name)
        if not sm:
            return None
        out = {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(seen),
               "samples": len(sm)}
        if nearest:
            out["nearest_before"] = True
        return out


def gpu_id_for(device) -> str:
    import torch
    props = torch.cuda.get_device_properties(device)
    uuid = getattr(props, "uuid", None)
    if uuid:
        s = str(uuid)
        return s if s.startswith("GPU-") else "GPU-" + s
    return str(device.index or 0)


def clocks_rejected(c: dict | None) -> bool:
    if not c:
        return False
    if any(r in c["reasons"] for r in REJECT):
        return True
    return c["sm_mhz"] < 0.6 * c["sm_max_mhz"] and not c["reasons"]


# ---- peaks and profiles -----------------------------------------------------
def hbm_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def gather_source_hash() -> str:
    with open(GATHER_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(workload: str) -> tuple[float | None, str | None]:
    """DRAM bytes per gather row position from the committed ncu summary, if
    it was taken on the current gather.cu (else None); the caller scales it
    to its launch."""
    path = os.path.join(PROFILES, f"gather_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None, None
    m = re.search(r"traffic_bytes_per_position:\s*([0-9.eE+]+)\s+source:\s*([0-9a-f]+)", text)
    if not m or m.group(2) != gather_source_hash():
        return None, None
    return float(m.group(1)), os.path.relpath(path, ROOT)


# ---- the workload ---------------------------------------------------------
def make_workload(name: str):
    from corpus import make_preset
    t = time.time()
    c = make_preset(name)
    log(f"[bench] corpus {name}: {c.n_docs} docs, {c.n_tokens} tokens, {time.time() - t:.1f}s")
    return c


def recipe_kwargs(c) -> dict:
    return dict(stream_doc_begin=c.stream_doc_begin, stream_source=c.stream_source,
                source_weight=c.source_weight, stream_weight=c.stream_weight,
                source_heldout_bp=c.source_heldout_bp, T=c.T, B=c.B, max_steps=c.max_steps,
                seed=c.seed, hash_key=c.hash_key, drain=c.drain, pad_id=c.pad_id)


def variant_kwargs(c, name: str) -> dict:
    """Packer / oracle options of a bench variant."""
    if name == "heldout":
        return dict(heldout_only=True, drain=True)
    if name == "shuffled":
        return dict(window_segment=64, shuffle_rows=True)
    if name == "wrap":
        return dict(wrap=True, len_bucket=256)
    if name == "schedule":
        rng = np.random.default_rng(77)
        K, B = int(c.max_steps), int(c.B)
        begins = sorted({0, K // 8, K // 4, K // 2})
        Bs = [max(1, B * (i + 1) // 4) for i in range(4)][-len(begins):]
        sw = np.asarray(c.source_weight, np.float64)
        tw = np.asarray(c.stream_weight, np.float64)
        return dict(schedule=[
            dict(begin=b, B=bb,
                 source_weight=np.maximum(1, np.rint(sw * rng.uniform(0.8, 1.25, sw.size)))
                 .astype(np.uint32).tolist(),
                 stream_weight=np.maximum(1, np.rint(tw * rng.uniform(0.8, 1.25, tw.size)))
                 .astype(np.uint32).tolist())
            for b, bb in zip(begins, Bs)])
    return {}


def auto_launch(max_steps: int, rows: int, T: int) -> int:
    """Most updates a launch takes: the horizon in equal launches of at most
    2^30 positions (a 14 GB output buffer; the longer a launch, the less its
    tail of partly idle SMs costs).  500 for the 512 x 4096 rows (1000
    updates), 200 for 256 x 8192 (200), 512 for 64 x 32768 (a horizon of
    1024, of which launch_plan splits the 574 valid updates into two of
    287), the whole horizon for 8 x 4096."""
    per = max(1, (1 << 30) // max(1, rows * T))
    n = -(-max_steps // per)
    return max(1, -(-max_steps // max(1, n)))


def launch_plan(pk, valid: int, L: int):
    """(first update, updates, rows per update) of each launch: at most L
    updates, never across a schedule piece (rows per update may change);
    each piece in launches of equal size (the fewest that fit L), so that
    no short launch is left at its end."""
    begins = sorted({int(p["begin"]) for p in pk.schedule}) if pk.schedule else [0]
    s = 0
    for e in [b for b in begins if 0 < b < valid] + [valid]:
        n = -(-(e - s) // L)
        per = -(-(e - s) // max(1, n))
        while s < e:
            m = min(per, e - s)
            yield s, m, pk.rows_of_step(s)
            s += m


def config_block(c, args, dist: Dist, rows, name: str) -> dict:
    return {"workload": f"{name}: {WORKLOADS[name]}",
            "variant": f"{args.variant}: {VARIANTS[args.variant]}",
            "n_docs": c.n_docs, "n_tokens": c.n_tokens, "T": c.T, "B": c.B,
            "updates_per_step": None, "rows_per_rank": rows[1] - rows[0],
            "launch_updates": args.launch, "row_slices_per_launch": args.slices,
            "l2": ("inputs larger than L2 (corpus %.1f GB, output buffer > 129 MB)"
                   % (c.n_tokens * 4 / 1e9)) if c.n_tokens * 4 > L2_BYTES else
                  ("corpus (%.3f GB) fits in L2: no flush between passes, a latency figure"
                   % (c.n_tokens * 4 / 1e9)),
            "parallelism": f"rows split over {dist.world} GPU(s), tables replicated"}


# ---- multi-rank bookkeeping (the path's only collectives) -----------------
def fold_runs(plan) -> list:
    """(first update, updates, rows per update) runs of consecutive launches
    with the same rows per update."""
    runs = []
    for s0, m, Bk in plan:
        if runs and runs[-1][2] == Bk and runs[-1][0] + runs[-1][1] == s0:
            runs[-1][1] += m
        else:
            runs.append([s0, m, Bk])
    return runs


def gather_batch_rows(dist: Dist, local, runs, world: int) -> list:
    """Row fingerprints of every update in global row order.  ``local`` is
    this rank's [updates, rows_max] tensor (its slice of every update's rows,
    padded to the largest slice); every rank's is gathered, then each run of
    updates with the same rows is put together slice after slice.  Returns one
    [updates, rows] tensor per run."""
    import torch
    if world == 1:
        parts = [local.unsqueeze(0)]
    else:
        parts = [torch.empty_like(local) for _ in range(world)]
        dist.pg.all_gather(parts, local)
        parts = [p.unsqueeze(0) for p in parts]
    allr = torch.cat(parts)  # [world, updates, rows_max]
    out = []
    for f0, fm, Bk in runs:
        cols = [allr[q, f0:f0 + fm, :row_slice(q, world, Bk)[1] - row_slice(q, world, Bk)[0]]
                for q in range(world)]
        out.append(torch.cat(cols, dim=1).contiguous())
    return out


def reduce_learned(dist: Dist, learned) -> None:
    """Every update's learned positions: each rank holds its slice's share;
    the update's count is their sum (in place)."""
    if dist.pg is not None:
        dist.pg.all_reduce(learned, op=dist.pg.ReduceOp.SUM)


# ---- our arm ----------------------------------------------------------------
def measure(args, dist: Dist, name: str, *, e2e: bool, cpu: bool, steps: int,
            warmup: int) -> dict | None:
    """Time whole passes of workload `name`; the JSON result on rank 0."""
    import torch
    from deterministic_packed_assembly_gb300 import Packer

    device = torch.device("cuda", dist.local)
    torch.cuda.set_device(device)
    c = make_workload(name)
    rows = row_slice(dist.rank, dist.world, c.B)
    rk = recipe_kwargs(c)
    rk.update(variant_kwargs(c, args.variant))
    stream = torch.cuda.current_stream(device)

    tok_d = torch.from_numpy(c.tokens).to(device)
    off_d = torch.from_numpy(c.doc_offsets).to(device)
    ls_d = None if c.loss_start is None else torch.from_numpy(c.loss_start).to(device)
    torch.cuda.synchronize()

    n_buf = -(-c.B // dist.world)  # bounds this rank's rows of any update
    L = args.launch or auto_launch(c.max_steps, n_buf, c.T)
    n_pos = L * n_buf * c.T
    # flat buffers, viewed [updates][rows][T] per launch (a schedule changes
    # the rows per update)
    out = dict(tokens=torch.empty(n_pos, dtype=torch.int32, device=device),
               pos=torch.empty(n_pos, dtype=torch.int32, device=device),
               doc=torch.empty(n_pos, dtype=torch.int32, device=device),
               mask=torch.empty(n_pos, dtype=torch.uint8, device=device))
    # every update's row fingerprints and learned counts stay for the pass
    # (8 + 4 bytes a row); the batch fingerprints of all updates are folded at
    # the end, one launch per run of updates with the same rows
    row_fp_all = torch.empty(c.max_steps * n_buf, dtype=torch.int64, device=device)
    row_ln_all = torch.empty(c.max_steps * n_buf, dtype=torch.int32, device=device)
    fp_all = torch.empty(c.max_steps, dtype=torch.int64, device=device)
    learned_all = torch.empty(c.max_steps, dtype=torch.int64, device=device)
    # with several ranks: this rank's row fingerprints of every update,
    # padded to n_buf rows, for the gather
    fp_local = (torch.zeros((c.max_steps, n_buf), dtype=torch.int64, device=device)
                if dist.world > 1 else None)

    state = {"launches": 0, "init_launches": 0, "valid": 0, "events": [], "rows_total": 0,
             "init_events": [], "hash_ns": []}
    # every pass has the same launch plan: each launch's views of the buffers
    # and their C description are built once, so that the first gather goes
    # out as soon as init returns
    launch_cache = {}
    # timing events, created before the timed region (one pair per init and
    # per launch of every timed pass)
    ev_pool = {"events": [], "i": 0}

    def next_event():
        if ev_pool["i"] == len(ev_pool["events"]):
            ev_pool["events"].append(torch.cuda.Event(enable_timing=True))
        ev_pool["i"] += 1
        return ev_pool["events"][ev_pool["i"] - 1]

    def one_pass(record: bool, count: bool = False, e2e_bufs=None):
        """One whole pass; returns real tokens assembled when `count`."""
        if record:
            ei0, ei1 = next_event(), next_event()
            ei0.record(stream)
        src = (tok_d, off_d, ls_d) if e2e_bufs is None else e2e_bufs[:3]
        pk = Packer(*src, stream=stream, device=device, **rk)
        if record:
            ei1.record(stream)
            state["init_events"].append((ei0, ei1))
        valid = pk.valid_steps
        state["valid"] = valid
        state["info"] = pk.info
        if record:
            state["hash_ns"].append(pk.info["hash_ns"])
        real = torch.zeros((), dtype=torch.int64, device=device) if count else None
        n = 0
        rows_total = 0
        plan = list(launch_plan(pk, valid, L))
        folds = []  # [first update, updates, rows, offset of their first row]
        for s0, m, Bk in plan:
            rk0, rk1 = row_slice(dist.rank, dist.world, Bk)
            r = rk1 - rk0
            if r == 0:
                continue
            ro = rows_total
            rows_total += m * r
            if folds and folds[-1][2] == r and folds[-1][0] + folds[-1][1] == s0:
                folds[-1][1] += m
            else:
                folds.append([s0, m, r, ro])
            key = (s0, m, r, ro)
            if key not in launch_cache:
                view = {k: v[:m * r * c.T].view(m, r, c.T) for k, v in out.items()}
                view["row_fp"] = row_fp_all[ro:ro + m * r].view(m, r)
                view["row_learned"] = row_ln_all[ro:ro + m * r].view(m, r)
                launch_cache[key] = (view, Packer.prepare(view))
            view, prepared = launch_cache[key]
            if record:
                ea, eb = next_event(), next_event()
                ea.record(stream)
            if args.slices <= 1:
                pk.step(s0, m, rows=(rk0, rk1), out=view, stream=stream, prepared=prepared)
                n += 1
            else:
                # R launches of row slices, each into its own contiguous region
                for si in range(args.slices):
                    a, e = row_slice(si, args.slices, r)
                    if e == a:
                        continue
                    vs = {k: v[m * a * c.T:m * e * c.T].view(m, e - a, c.T) for k, v in out.items()}
                    vs["row_fp"] = row_fp_all[ro + m * a:ro + m * e].view(m, e - a)
                    vs["row_learned"] = row_ln_all[ro + m * a:ro + m * e].view(m, e - a)
                    pk.step(s0, m, rows=(rk0 + a, rk0 + e), out=vs, stream=stream)
                    n += 1
            if record:
                eb.record(stream)
                state["events"].append((ea, eb))
            if count:
                real += (view["doc"] >= 0).sum()
        # each update's learned positions (this rank's share of them), and the
        # batch fingerprints of every update (row slices are not in batch
        # order, so they are skipped with --slices)
        if args.slices <= 1:
            for f0, fm, fr, fo in folds:
                pk.step_learned(row_ln_all[fo:fo + fm * fr].view(fm, fr),
                                out=learned_all[f0:f0 + fm], stream=stream)
                n += 1
            if dist.world == 1:
                for f0, fm, fr, fo in folds:
                    pk.batch_fp_many(row_fp_all[fo:fo + fm * fr].view(fm, fr),
                                     out=fp_all[f0:f0 + fm], stream=stream)
                    n += 1
            else:
                # the two collectives of a row split: the learned counts
                # summed over ranks, the row fingerprints gathered in row
                # order and folded into every update's batch fingerprint
                reduce_learned(dist, learned_all[:valid])
                for f0, fm, fr, fo in folds:
                    fp_local[f0:f0 + fm, :fr].copy_(row_fp_all[fo:fo + fm * fr].view(fm, fr))
                runs = fold_runs(plan)
                for (f0, fm, _), rows_k in zip(runs, gather_batch_rows(dist, fp_local[:valid],
                                                                       runs, dist.world)):
                    pk.batch_fp_many(rows_k, out=fp_all[f0:f0 + fm], stream=stream)
                    n += 1
        if e2e_bufs is not None:
            e2e_bufs[3][:rows_total].copy_(row_fp_all[:rows_total], non_blocking=True)
            e2e_bufs[4][:rows_total].copy_(row_ln_all[:rows_total], non_blocking=True)
            e2e_bufs[5][:valid].copy_(fp_all[:valid], non_blocking=True)
            e2e_bufs[6][:valid].copy_(learned_all[:valid], non_blocking=True)
        pk.close()
        state["launches"] = n
        state["rows_total"] = rows_total
        return int(real.item()) if count else None

    # warm-up (the first pass also counts the real tokens of a pass)
    real_tokens = one_pass(False, count=True)
    for _ in range(max(warmup - 1, 0)):
        one_pass(False)
    valid = state["valid"]
    rows_pass = state["rows_total"]  # rows this rank assembles in a pass
    positions = rows_pass * c.T
    log(f"[bench] {name} rank {dist.rank}: {valid} updates, {real_tokens} real tokens / pass")

    def timed(K: int):
        state["events"].clear()
        state["init_events"].clear()
        state["hash_ns"].clear()
        n_ev = 2 * K * (len(launch_cache) * max(args.slices, 1) + 1)
        while len(ev_pool["events"]) < n_ev:
            ev_pool["events"].append(torch.cuda.Event(enable_timing=True))
        ev_pool["i"] = 0
        sampler = ClockSampler(gpu_id_for(device)) if dist.rank == 0 else None
        dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if sampler:
            sampler.mark()
        t0.record(stream)
        for _ in range(K):
            one_pass(True)
        t1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        clocks = sampler.stop() if sampler else None
        ms = t0.elapsed_time(t1)
        gather_ms = [a.elapsed_time(b) for a, b in state["events"]]
        state["init_ms"] = float(np.mean([a.elapsed_time(b) for a, b in state["init_events"]]))
        return ms, gather_ms, clocks

    K = steps
    ms, gather_ms, clocks = timed(K)
    retried = False
    if clocks_rejected(clocks):
        log(f"[bench] clocks rejected ({clocks}); measuring once more")
        ms, gather_ms, clocks = timed(K)
        retried = True
    ms_max = dist.max(ms)
    total_real = dist.sum(real_tokens) * K
    value = total_real / (ms_max / 1e3)

    # roofline of the gather kernel: algorithmic bytes per launch / its time
    n_launch = len(gather_ms) // K
    alg_gather = 13.0 * positions + 4.0 * real_tokens + 12.0 * rows_pass
    bytes_per_launch = alg_gather / n_launch
    avg_launch_s = (sum(gather_ms) / len(gather_ms)) / 1e3
    peak, peak_kind = hbm_peak()
    achieved = bytes_per_launch / avg_launch_s / 1e9
    traffic_pp, traffic_src = profiled_traffic(name)
    # per launch, like `achieved`: the captured launch's bytes per position
    # times this launch's positions (traffic grows with positions)
    traffic = None if traffic_pp is None else traffic_pp * positions / n_launch
    gather_share = sum(gather_ms) / ms
    info = state["info"]

    # collectives first: every rank takes part
    alg_gather_all = dist.sum(alg_gather)
    positions_all = dist.sum(positions)
    result = None
    if dist.rank == 0:
        # the pass's algorithmic bytes: the gather's, plus what the held-out
        # hash read as the library counted it (4 B a token, 8 B of offsets a
        # document; every rank hashes the same prefix)
        hashed_bytes = 4.0 * info["hashed_tokens"] + 8.0 * info["hashed_docs"]
        alg_step = alg_gather_all + hashed_bytes
        cfg = config_block(c, args, dist, rows, name)
        cfg["updates_per_step"] = valid
        cfg["launch_updates"] = L
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": K,
            "warmup": warmup, "ms_per_step": ms_max / K, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "int32",
            "data": f"synthetic (numpy PCG64, data seed {c.notes.get('data_seed')})",
            "config": cfg,
            "positions_per_s": positions_all * K / (ms_max / 1e3),
            "init_ms_per_step": state["init_ms"],
            "alg_gbps_step": alg_step * K / (ms_max / 1e3) / 1e9,
            "alg_bytes_step": {"gather": alg_gather_all, "hash": hashed_bytes,
                               "hashed_tokens": info["hashed_tokens"],
                               "hashed_docs": info["hashed_docs"],
                               "note": "hash: the tokens and documents the library's hash "
                                       "kernel counted it read (4 B a token, 8 B of offsets "
                                       "a document)"},
            "roofline": {"kernel": "gather_kernel", "bound": "hbm", "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "traffic": traffic,
                         "traffic_source": traffic_src,
                         "bytes_per_launch": bytes_per_launch,
                         "avg_launch_ms": avg_launch_s * 1e3, "launches": len(gather_ms),
                         "share_of_step": gather_share},
            "gpu_launches": K * (info["init_launches"] + state["launches"]),
            "clocks": clocks, "clocks_retried": retried,
        }
        if info["hashed_tokens"] and state["hash_ns"]:
            result["hash_roofline"] = hash_roofline(info["hashed_tokens"],
                                                    float(np.mean(state["hash_ns"])) * 1e-9,
                                                    device, stream)

    # ---- end to end: host inputs, copies inside the timed region -----------
    if e2e:
        tok_h = torch.from_numpy(c.tokens).pin_memory()
        off_h = torch.from_numpy(c.doc_offsets).pin_memory()
        ls_h = None if c.loss_start is None else torch.from_numpy(c.loss_start).pin_memory()
        fp_h = torch.empty(c.max_steps * n_buf, dtype=torch.int64).pin_memory()
        ln_h = torch.empty(c.max_steps * n_buf, dtype=torch.int32).pin_memory()
        bf_h = torch.empty(c.max_steps, dtype=torch.int64).pin_memory()
        sl_h = torch.empty(c.max_steps, dtype=torch.int64).pin_memory()

        def e2e_pass():
            # the corpus goes to the library in page-locked host memory: it
            # reads the documents the horizon reaches where they lie (the hash
            # writes what it reads into its device copy) and copies nothing
            # else
            one_pass(False, e2e_bufs=(tok_h, off_h, ls_h, fp_h, ln_h, bf_h, sl_h))

        # two untimed passes: the first reads of page-locked memory over the
        # host link settle in only after a pass or two
        e2e_pass()
        e2e_pass()
        dist.barrier()
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_pass()
        torch.cuda.synchronize()
        e2e_s = dist.max(time.perf_counter() - t)
        # bytes the library read from host memory (offsets, loss starts, the
        # tokens of the documents it used), as it reports them
        h2d = int(state["info"]["host_bytes"])
        d2h = rows_pass * 12 + valid * 8 + valid * 8
        if result is not None:
            result["e2e"] = {"value": dist.sum(real_tokens) * args.e2e_steps / e2e_s,
                             "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                             "steps": args.e2e_steps,
                             "corpus_bytes": tok_h.numel() * 4 + off_h.numel() * 8
                             + (0 if ls_h is None else ls_h.numel() * 4),
                             "path": "Packer (C ABI, NS_PACK_HOST_CORPUS) on page-locked host "
                                     "inputs: the library reads the documents the horizon "
                                     "reaches from host memory (hash and prefix copy write "
                                     "them to its device copy), full pass; the [B, T] batches "
                                     "stay resident on the device for a trainer on the same "
                                     "GPU, and every row fingerprint and learned count and "
                                     "every update's batch fingerprint and learned positions "
                                     "are copied back to the host"}
        else:
            dist.sum(real_tokens)

    # ---- CPU baseline: the oracle on one measured pass (rank 0, N=1) -------
    if result is not None and cpu and dist.world == 1 and args.slices <= 1:
        fp_gpu = fp_all[:valid].cpu().numpy().view(np.uint64)
        result["cpu_baseline"] = cpu_baseline(c, args, valid, real_tokens, fp_gpu,
                                              variant_kwargs(c, args.variant))
    del out, tok_d, off_d, ls_d, row_fp_all, row_ln_all
    torch.cuda.empty_cache()
    return result


def hash_roofline(tokens: int, seconds: float, device, stream) -> dict:
    """The held-out hash against its integer ceiling: tokens hashed per
    second inside the pass (its phase of init, both rounds, timed by the
    library with CUDA events) over the rate of a register-only loop of the
    same per-token term (ns_pack_probe_hash_terms), timed here."""
    import torch
    import deterministic_packed_assembly_gb300 as nsp
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    blocks, per = sms * 8, 8192
    acc = torch.zeros(1, dtype=torch.int64, device=device)
    nsp.ns_pack_probe_hash_terms(blocks, per, acc.data_ptr(), stream.cuda_stream)
    best = None
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        nsp.ns_pack_probe_hash_terms(blocks, per, acc.data_ptr(), stream.cuda_stream)
        b.record(stream)
        b.synchronize()
        t = a.elapsed_time(b) / 1e3
        best = t if best is None else min(best, t)
    peak = blocks * 256 * per / best
    achieved = tokens / seconds
    return {"kernel": "hash_prefix_kernel", "bound": "alu", "achieved": achieved,
            "peak": peak, "unit": "terms/s", "frac": achieved / peak,
            "peak_kind": "measured: register-only loop of the same per-token term "
                         "(ns_pack_probe_hash_terms, %d x 256 threads x %d terms)" % (blocks, per),
            "tokens": tokens, "ms": seconds * 1e3}


def run_ours(args, dist: Dist) -> None:
    result = measure(args, dist, args.config, e2e=not args.no_e2e, cpu=not args.no_cpu_baseline,
                     steps=args.steps, warmup=args.warmup)
    # the other workloads named with it, each timed the same way (GPU pass,
    # gather roofline, e2e); no CPU baseline
    extra = {}
    for name in [x for x in args.also.split(",") if x and x not in ("none", args.config)]:
        # four times the steps: a pass of these is a few ms, and the clock
        # sampler needs a timed region of a few of its 50 ms periods
        r = measure(args, dist, name, e2e=not args.no_e2e, cpu=False,
                    steps=4 * args.steps, warmup=max(3, min(args.warmup, 3)))
        if r is not None:
            extra[name] = {k: r[k] for k in ("value", "unit", "steps", "warmup", "ms_per_step",
                                             "config", "positions_per_s", "init_ms_per_step",
                                             "alg_gbps_step", "alg_bytes_step", "roofline",
                                             "gpu_launches", "clocks", "e2e") if k in r}
    if result is not None:
        if extra:
            result["extra_configs"] = extra
        print(json.dumps(result), flush=True)


def cpu_baseline(c, args, valid: int, real_tokens: int, fp_gpu=None, vk=None) -> dict:
    """Time the oracle as it stands (one host thread) on one whole pass of the
    workload: its build (hash, shuffle, pack, quotas over the whole corpus)
    and the rows of every valid update, measured, nothing scaled.  With the
    GPU's batch fingerprints it also checks every update bit for bit."""
    import oracle
    t = time.perf_counter()
    o = oracle.Oracle(c, **(vk or {}))
    t_build = time.perf_counter() - t
    fps = []
    t = time.perf_counter()
    for k in range(valid):
        fps.append(oracle.batch_fp(o.rows(k)["row_fp"]))
    t_rows = time.perf_counter() - t
    t_full = t_build + t_rows
    out = {"value": real_tokens / t_full, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"one whole pass, measured: oracle build over the whole corpus "
                     f"({t_build:.2f} s) + the rows of all {valid} updates ({t_rows:.2f} s)",
           "extrapolated": False, "build_s": t_build, "rows_s": t_rows}
    if fp_gpu is not None:
        out["bit_exact_updates"] = int(sum(int(fp_gpu[k]) == fps[k] for k in range(valid)))
        out["bit_exact_all"] = bool(out["bit_exact_updates"] == valid)
        out["valid_steps_match"] = bool(o.valid_steps == valid)
    return out


# ---- reference arm: the oracle --------------------------------------------
REFERENCE_BUDGET_S = 180.0  # timed oracle passes stop once they pass this


def run_reference(args, dist: Dist) -> None:
    if dist.rank != 0:
        return
    import oracle
    oracle.build()
    c = make_workload(args.config)
    vk = variant_kwargs(c, args.variant)

    def ref_pass(count: bool = False):
        """One whole pass of the oracle: build, then every update's rows;
        with `count`, also the real (non-pad) tokens it assembled."""
        t = time.perf_counter()
        oo = oracle.Oracle(c, **vk)
        real = 0
        for k in range(oo.valid_steps):
            r = oo.rows(k)
            if count:
                real += int((r["doc"] >= 0).sum())
        return time.perf_counter() - t, real, oo.valid_steps

    # a CPU program needs no warm-up beyond one pass (which also counts the
    # pass's real tokens, untimed); the timed passes stop once
    # REFERENCE_BUDGET_S is spent (at least two), so that the run ends within
    # a few minutes: the counts run are the ones reported
    _, real, valid = ref_pass(count=True)
    warm = 1
    times = []
    t_start = time.perf_counter()
    while len(times) < args.steps:
        times.append(ref_pass()[0])
        if len(times) >= 2 and time.perf_counter() - t_start > REFERENCE_BUDGET_S:
            break
    step_s = float(np.mean(times))
    value = real / step_s
    sample = (f"each step one whole oracle pass, measured: build over the whole corpus + the "
              f"rows of all {valid} updates; {len(times)} of {args.steps} requested steps "
              f"timed (budget {REFERENCE_BUDGET_S:.0f} s), {warm} warm-up pass(es)")
    rows = (0, c.B)
    result = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": dist.world, "steps": len(times), "steps_requested": args.steps,
        "warmup": warm, "warmup_requested": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "int32",
        "data": f"synthetic (numpy PCG64, data seed {c.notes.get('data_seed')})",
        "config": dict(config_block(c, args, dist, rows, args.config), updates_per_step=valid),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


def main():
    args = parse_args()
    dist = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
