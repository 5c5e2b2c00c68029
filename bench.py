"""Benchmark of the sparse-embedding training step on GB300.

Workload: Criteo-shaped DLRM embedding layer -- 26 fp32 tables of dim 128 (8 tables of 10M
rows, 18 tables log-spaced 100..1M rows, 82.4M rows, 42 GB of parameters + 42 GB of
Adagrad accumulators), batch 65536, one Zipf(1.05) ID per (sample, table) through a seeded
permutation of ranks, 27-vector dot interaction with a dense N(0,1) vector, N(0,1)
upstream gradient, per-element Adagrad.  Synthetic inputs stand in for the Criteo click
logs.  One step = lookup + dedup + gather + interaction forward, interaction backward +
per-unique-row gradient reduction + Adagrad on the touched rows.

Output: one JSON line (rank 0).  `value` is samples/s over all ranks with the inputs
resident in HBM; `e2e` repeats the measurement through the host-buffer entry point with
the copies in the timed region; `roofline` reports the dominant kernel against the
measured HBM bandwidth; `cpu_baseline` times the CPU oracle on a bounded sample.
`--impl reference` times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "embedding fwd+bwd+Adagrad samples/s; achieved HBM GB/s as % of GB300 peak"
UNIT = "samples/s"
FALLBACK_HBM_GBS = 6800.0
NUM_BATCHES = 3  # distinct seeded batches, used round robin


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # about a second of timed steps on the default workload, so that the clock sampler (one
    # reading per 200 ms) covers the timed region several times
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-sample", type=int, default=2048)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--small", action="store_true", help="shrunken tables/batch (for smoke runs)")
    ap.add_argument("--rows-div", type=int, default=1,
                    help="divide every table's rows by this (profiling captures on a few GB)")
    ap.add_argument("--admit", type=int, default=-1,
                    help="hashed workload: admission minimum (turns on per-key counts)")
    ap.add_argument("--tier-cache", type=int, default=0,
                    help="static workloads: keep the tables in the host tier with an HBM cache "
                         "of this many rows (a power of two)")
    ap.add_argument("--tier-prefetch", action="store_true",
                    help="tiered: prefetch the next batch's rows on a second stream during each step")
    ap.add_argument("--tier-watermark", type=str, default="",
                    help="tiered: HIGH,LOW cache rows for the watermark check after every step")
    ap.add_argument("--evict-every", type=int, default=0,
                    help="hashed (with --admit) or tiered workloads: evict after every K-th step")
    ap.add_argument("--evict-idle", type=int, default=4,
                    help="eviction: keys idle for more than this many steps")
    ap.add_argument("--evict-min", type=int, default=0,
                    help="eviction: keys counted fewer than this many times")
    ap.add_argument("--cross", action="store_true",
                    help="time the cross interaction layer (forward + backward) on one batch")
    ap.add_argument("--codec", action="store_true",
                    help="time the int8 row codec (encode + decode) on one batch of pooled rows")
    ap.add_argument("--batch", type=int, default=0,
                    help="samples per batch instead of the workload's (profiling captures)")
    ap.add_argument("--config", type=int, default=2, choices=[2, 3, 4, 5],
                    help="workload: 2 Criteo-shaped fused step (default), 3 multi-hot bf16 "
                         "mean-pooled row-wise Adagrad, 4 hashed dynamic table (its 20 fixed "
                         "steps), 5 uniform bandwidth stress")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def sync_ranks(ws: int):
    """Barrier across the replicas (no-op on one rank)."""
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ms: float, ws: int, device) -> float:
    """The timed region's length as the slowest replica measured it (every rank calls this)."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, ws: int, steps: int, ms: float) -> float:
    """Units all replicas processed per second over the slowest replica's time."""
    return ws * units_per_rank * steps / (ms / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def workload(small: bool, rows_div: int = 1, config: int = 2, batch: int = 0):
    import dataclasses
    import synth
    w = synth.workload(config, "small" if small else "full")
    if rows_div > 1 and w.rows is not None:
        w = dataclasses.replace(w, rows=[max(100, r // rows_div) for r in w.rows],
                                name=f"{w.name}-rows-div{rows_div}")
    if batch > 0:
        w = dataclasses.replace(w, batch=batch, name=f"{w.name}-batch{batch}")
    return w


# ------------------------------------------------------------------ CPU oracle timing

def num_batches(w) -> int:
    """Distinct seeded batches the timed steps cycle through: the hashed workload runs its
    fixed sequence of steps (new keys arrive over time), the others rotate three batches."""
    return w.steps if w.hashed else NUM_BATCHES


def oracle_step(orc, w, b, S: int):
    """The oracle's full step on the first S samples of batch b."""
    import oracle
    T, D = w.num_tables, w.dim
    if b.offsets is None:
        ids, offs = b.ids[: S * T], None
    else:
        offs = b.offsets[: S * T + 1]
        ids = b.ids[: int(offs[-1])]
    pooled, pmag, _ = orc.forward(ids, offs, S)
    if w.interaction:
        dense, dout = b.dense[:S], b.dout[:S]
        oracle.interact(dense, pooled, T, D, pmag)
        _, dp, _, mp = oracle.interact_backward(dout, dense, pooled, T, D, pmag)
        orc.backward_adagrad(dp, mp)
    else:
        g = b.dout[:S].astype(np.float64)
        orc.backward_adagrad(g, np.abs(g))


def host_cores() -> int:
    return os.cpu_count() or 1


def time_oracle(w, batches, seconds: float, sample: int, min_steps: int = 1, max_steps: int = 10**9):
    """Run the oracle's full step on the first `sample` samples of successive batches until
    `seconds` of CPU time have passed (at least min_steps), pinned to one host core (the
    oracle is single-threaded).  Returns (samples/s, steps, s)."""
    import oracle
    orc = oracle.Model.from_workload(w)
    done, t_total, k = 0, 0.0, 0
    old = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    if old:
        os.sched_setaffinity(0, {min(old)})
    try:
        while (t_total < seconds or k < min_steps) and k < max_steps:
            b = batches[k % len(batches)]
            S = min(sample, b.batch)
            t0 = time.perf_counter()
            oracle_step(orc, w, b, S)
            t_total += time.perf_counter() - t0
            done += S
            k += 1
    finally:
        if old:
            os.sched_setaffinity(0, old)
    return (done / t_total if t_total > 0 else 0.0), k, t_total


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import synth
    w = workload(args.small, args.rows_div, args.config, args.batch)
    batches = [synth.make_batch(w, s) for s in range(min(num_batches(w), args.steps + args.warmup))]
    # each step is a bounded sample of the workload, sized so that the whole run (warm-up and
    # timed steps) stays within about a minute of single-core oracle time at any K
    S = min(args.cpu_sample, w.batch, max(32, int(2.5e5 / (args.steps + args.warmup))))
    time_oracle(w, batches, 0.0, S, min_steps=args.warmup, max_steps=args.warmup)
    v, k, secs = time_oracle(w, batches, 0.0, S, min_steps=args.steps, max_steps=args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(k, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {**workload_config(w), "global_batch": w.batch, "parallelism": "none"},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "host_cores": host_cores(),
                         "kind": "oracle",
                         "sample": f"first {S} samples of each {w.batch}-sample batch, full step, "
                                   f"single thread pinned to one of the host's {host_cores()} cores"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        self.path = os.path.join("/tmp", f"emb_clocks_{os.getpid()}.csv")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(device)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        try:
            rows = [l.strip().split(",") for l in open(self.path) if l.strip()]
            os.remove(self.path)
        except Exception:
            return None
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            if len(r) < 9:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        top = max(sm)
        loaded = [s for s in sm if s >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_config(w) -> dict:
    """The `config` description of a workload (shapes and input recipe)."""
    c = {"workload": w.name, "tables": w.num_tables, "dim": w.dim, "dtype": w.dtype,
         "ids": {"zipf": f"zipf({w.alpha}) over a seeded permutation of ranks",
                 "zipf_keys": f"zipf({w.alpha}) over {w.num_keys} keys (63-bit bijection)",
                 "uniform": "uniform"}[w.ids_dist],
         "bags": {"one": "one id per (sample, table)", "poisson": f"min(1+Poisson({w.bag_mu}), {w.bag_cap})",
                  "uniform_1_4": "uniform 1..4"}[w.bag],
         "pooling": w.pooling,
         "optimizer": f"{w.optimizer}, lr {w.lr}, eps {w.eps}, acc0 {w.init_acc}"}
    if w.hashed:
        c["hash_capacity"] = w.capacity
        c["steps_cycled"] = w.steps
    else:
        c["rows_total"] = int(sum(w.rows))
    if w.interaction:
        c["interaction"] = f"{w.num_features} vectors -> {w.num_pairs} pairs + {w.dim} dense"
    return c


def hashed_policy(w, args) -> dict:
    """Tiering, admission and eviction settings of a run (empty when not used)."""
    c = {}
    if not w.hashed and args.tier_cache > 0:
        c["tiered"] = (f"{int(sum(w.rows))} rows in the host tier (host-mapped memory), "
                       f"HBM cache of {args.tier_cache} rows")
    elif not w.hashed or args.admit < 0:
        return {}
    else:
        c["admission_min_count"] = args.admit
    if not w.hashed and args.tier_cache > 0:
        if args.tier_prefetch:
            c["prefetch"] = "next batch's rows on a second stream while each step runs"
        if args.tier_watermark:
            hi, lo = (int(x) for x in args.tier_watermark.split(","))
            c["watermark"] = f"after every step: over {hi} cached rows, evict the idlest to {lo}"
    if args.evict_every > 0:
        c["eviction"] = (f"after every {args.evict_every} steps: keys idle > {args.evict_idle} "
                         f"steps or counted < {args.evict_min} times")
    return c


# ------------------------------------------------------------------ algorithmic bytes

def kernel_bytes(w, U: int, L: int, once: int = 0):
    """Algorithmic bytes of one launch of each step kernel: L lookups, U unique rows, of
    which `once` rows (looked up once, in a step that tracks them) are updated by the
    interaction backward instead of the update kernel."""
    B, T, D = w.batch, w.num_tables, w.dim
    Wd = w.out_width
    row = 4 * D                                      # fp32 rows and gradients
    srow = 2 * D if w.dtype == "bf16" else 4 * D     # stored table rows
    acc = 4 if w.optimizer == "adagrad_row" else 4 * D
    bags = B * T
    return {
        # ids read, row/slot written (+ one probed key per lookup, hashed); dedup-set
        # traffic stays in L2
        "map_dedup": L * (8 + 4 + 4 + (8 if w.hashed else 0)) + U * 12,
        "expand_bags": bags * 4 + L * 4,
        # gathered rows + dense in, interaction out, per-lookup indices
        "fused_fwd": B * (T * row + row + 4 * Wd) + B * T * 16,
        # re-gathered rows, dense, dout in; d_dense out; per-unique gradient rows written
        # once; a once row instead: its acc row read, w and acc rows written
        "fused_bwd": B * (T * row + 2 * row + 4 * Wd) + B * T * 4 + (U - once) * row
                     + once * 3 * row,
        # gathered rows and row indices in, pooled rows out
        "pool": L * (srow + 4) + bags * row,
        # lookup -> unique index and per-unique counts; prefix sums; sorted positions
        "inverse": L * 8 + (U if once else 0),
        "inverse_count": L * 8,
        "fill_perm": L * 12,
        # each lookup's pooled-gradient row in; per unique row w and acc read + written
        # (one-hot), or its gradient row written to g (multi-hot: the update follows)
        "segreduce_adagrad": L * (row + 8) + (U * row if w.multi_hot else U * (2 * srow + 2 * acc)),
        # per unique row: g read + zeroed, w and acc read + written, its indices read and
        # its set key freed; in a step with once rows, only the other rows (listed)
        "adagrad_from_g": (U - once) * (2 * row + 2 * srow + 2 * acc) + (U - once) * 12,
        # per unique row: once flag and slot read; once rows: key freed, flag cleared; other
        # rows: row read, (u, row, slot) listed
        "once_split": U * 5 + once * 5 + (U - once) * 16,
        # per unique key: slot and count read, packed count/step read and written, hold flag
        "admit": U * 25,
        # per slot: key and packed count/step read (evicted slots also rewrite their key,
        # counters, row and accumulator; not counted: their number varies by step)
        "evict": (w.capacity or 0) * 16,
        # tiered: per row brought into the cache, its row and accumulator read from the host
        # tier and written to HBM (upper bound: every unique row of the batch)
        "tier_fill": U * 2 * (srow + acc),
    }


def traffic_for(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if its kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        d = json.load(open(path))
        ent = d[kernel]
        src = os.path.join(ROOT, ent["source"])
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if sha != ent["source_sha256"]:
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ our arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)

    import synth
    import recommender_model_embedding_gb300 as E

    w = workload(args.small, args.rows_div, args.config, args.batch)
    B, T, D = w.batch, w.num_tables, w.dim
    Wd = w.out_width
    nbat = num_batches(w)
    host_batches = [synth.make_batch(w, s) for s in range(nbat)]
    dev_t = lambda a: None if a is None else torch.from_numpy(a).to(dev)
    batches = [dict(ids=dev_t(hb.ids), offs=dev_t(hb.offsets), dense=dev_t(hb.dense),
                    dout=dev_t(hb.dout), nnz=int(hb.ids.size)) for hb in host_batches]
    L_max = max(bt["nnz"] for bt in batches)
    ctx = E.EmbCtx.from_workload(w, max_batch=B, max_lookups=max(L_max, w.max_lookups()),
                                 cache_rows=0 if w.hashed else args.tier_cache)

    def maybe_evict(k):
        if args.evict_every > 0 and (k + 1) % args.evict_every == 0:
            ctx.evict(args.evict_idle, args.evict_min, wait=False)
    tiered = not w.hashed and args.tier_cache > 0
    side = torch.cuda.Stream(dev) if tiered and args.tier_prefetch else None
    if side is not None:
        side.wait_stream(torch.cuda.current_stream())  # the batches were copied there
    if tiered and args.tier_watermark:
        ctx.set_tier_watermark(*(int(x) for x in args.tier_watermark.split(",")))

    def maybe_prefetch(k):  # the next step's rows, while this step computes
        if side is not None:
            nb = batches[(k + 1) % nbat]
            ctx.prefetch(nb["ids"], nb["offs"], B, stream=side)
    stream = torch.cuda.current_stream()
    if w.interaction:
        out = torch.empty((B, Wd), device=dev)
        ddense = torch.empty((B, D), device=dev)

        def step(k):
            bt = batches[k % nbat]
            ctx.forward_interact(bt["ids"], bt["offs"], B, bt["dense"], out)
            maybe_prefetch(k)
            ctx.backward_interact_adagrad(bt["dout"], bt["dense"], ddense)
            maybe_evict(k)
    else:
        pooled = torch.empty((B, T, D), device=dev)

        def step(k):
            bt = batches[k % nbat]
            ctx.forward(bt["ids"], bt["offs"], B, pooled)
            maybe_prefetch(k)
            ctx.backward_adagrad(bt["dout"])
            maybe_evict(k)
    if w.hashed and args.admit >= 0:
        ctx.set_admission(args.admit)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    flags = ctx.get_status()
    if flags:
        raise RuntimeError(f"device flags after warm-up: {flags:#x}")

    # timed region: device events, kernel events (for the roofline) and clock sampling
    ctx.profile(True)
    ctx.profile_reset()
    clocks = ClockSampler(dev.index) if rank == 0 else None
    sync_ranks(ws)
    torch.cuda.synchronize()
    n0 = ctx.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for k in range(args.warmup, args.warmup + args.steps):
        step(k)
    ev1.record(stream)
    torch.cuda.synchronize()
    launches = ctx.launch_count() - n0
    ms = max_over_ranks(ev0.elapsed_time(ev1), ws, dev)
    sync_ranks(ws)
    clk = clocks.stop() if clocks else None
    prof = ctx.profile_read()
    ctx.profile(False)
    keys, counts = ctx.read_unique()  # unique rows of the last timed step
    U = int(keys.size)
    once_rows = int((counts == 1).sum()) if ctx.step_tracks_once() else 0
    L_last = batches[(args.warmup + args.steps - 1) % nbat]["nnz"]

    # end to end through the public API from pinned host buffers: the host-buffer step for
    # the interaction workloads; copies around forward + backward_adagrad otherwise
    e2e = None
    if not args.no_e2e:
        hb = host_batches[0]
        pin = lambda a: None if a is None else torch.from_numpy(a).pin_memory()
        h_ids, h_offs, h_dense, h_dout = pin(hb.ids), pin(hb.offsets), pin(hb.dense), pin(hb.dout)
        if w.interaction:
            h_out = torch.empty((B, Wd)).pin_memory()
            h_dd = torch.empty((B, D)).pin_memory()
            h2d = h_ids.numel() * 8 + h_dense.numel() * 4 + h_dout.numel() * 4
            d2h = h_out.numel() * 4 + h_dd.numel() * 4

            def host_step():
                ctx.train_step_host(h_ids, h_offs, B, h_dense, h_dout, h_out, h_dd)
        else:
            h_pooled = torch.empty((B, T, D)).pin_memory()
            d_ids = torch.empty_like(h_ids, device=dev)
            d_offs = None if h_offs is None else torch.empty_like(h_offs, device=dev)
            d_dout = torch.empty_like(h_dout, device=dev)
            h2d = h_ids.numel() * 8 + h_dout.numel() * 4 + (0 if h_offs is None else h_offs.numel() * 4)
            d2h = h_pooled.numel() * 4

            def host_step():
                d_ids.copy_(h_ids, non_blocking=True)
                if d_offs is not None:
                    d_offs.copy_(h_offs, non_blocking=True)
                d_dout.copy_(h_dout, non_blocking=True)
                ctx.forward(d_ids, d_offs, B, pooled)
                h_pooled.copy_(pooled, non_blocking=True)
                ctx.backward_adagrad(d_dout)
        for _ in range(2):
            host_step()
        torch.cuda.synchronize()
        sync_ranks(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            host_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), ws, dev)
        e2e = {"value": whole_job_rate(B, ws, args.e2e_steps, ems), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": ems / args.e2e_steps}

    flags = ctx.get_status()
    if rank != 0:
        ctx.close()
        if ws > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    kb = kernel_bytes(w, U, L_last, once_rows)
    per_kernel = {n: {"ms_per_launch": t / c, "launches": c} for n, (t, c) in prof.items()}
    dom = max((n for n in prof if n in kb), key=lambda n: prof[n][0])
    dom_ms = prof[dom][0] / prof[dom][1]
    achieved = kb[dom] / (dom_ms / 1e3) / 1e9
    traffic = (traffic_for(dom) if args.config == 2 and args.rows_div == 1 and not args.small
               and not args.batch else None)
    srow = (2 if w.dtype == "bf16" else 4) * D
    acc_b = 4 if w.optimizer == "adagrad_row" else 4 * D
    gathered = L_last * srow
    updated = U * (2 * srow + 2 * acc_b)
    step_s = ms / args.steps / 1e3
    in_bytes = sum(int(x.numel()) * x.element_size() for x in batches[0].values()
                   if isinstance(x, torch.Tensor))
    line = {
        "metric": METRIC,
        "value": whole_job_rate(B, ws, args.steps, ms),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {**workload_config(w), **hashed_policy(w, args), "global_batch": ws * B,
                   "per_gpu_batch": B,
                   "l2": (f"not flushed: inputs larger than L2 ({nbat} rotating batches, "
                          f"{in_bytes / 1e6:.0f} MB of step inputs and "
                          f"{gathered / 1e6:.0f} MB of gathered rows per step)"),
                   "parallelism": "replicas" if ws > 1 else "single"},
        "headline": {"bytes_per_step": gathered + updated, "gathered_bytes": gathered,
                     "updated_bytes": updated, "unique_rows": U,
                     "once_rows_updated_in_backward": once_rows,
                     "gbps": (gathered + updated) / step_s / 1e9,
                     "frac_of_peak": (gathered + updated) / step_s / 1e9 / peak,
                     "peak_gbps": peak, "peak_kind": peak_kind},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": kb[dom], "ms_per_launch": dom_ms,
                     "peak_kind": peak_kind},
        "kernels": per_kernel,
        "gpu_launches": int(launches),
        "clocks": clk,
        # the step time scaled to the maximum SM clock by the median clock sampled under load
        "ms_per_step_at_max_clock": (ms / args.steps * clk["sm_mhz"] / clk["sm_max_mhz"]
                                     if clk and clk.get("sm_max_mhz") else None),
        "e2e": e2e,
        "device_flags": flags,
    }
    if not args.no_cpu_baseline:
        S = min(args.cpu_sample, B)
        v, k, secs = time_oracle(w, host_batches, args.cpu_seconds, S)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "host_cores": host_cores(),
                                "kind": "oracle",
                                "sample": f"first {S} samples of the {B}-sample batches, full step, "
                                          f"{k} steps in {secs:.1f} s, single thread pinned to one "
                                          f"of the host's {host_cores()} cores"}
    print(json.dumps(line), flush=True)
    ctx.close()
    if ws > 1:
        dist.destroy_process_group()


def run_codec(args):
    """int8 row codec on the pooled rows of one batch of the workload (one GPU): encode and
    decode timed with CUDA events on the launching stream; the oracle timed on a sample."""
    import time
    import numpy as np
    import torch
    import recommender_model_embedding_gb300 as E
    w = workload(args.small, args.rows_div, args.config, args.batch)
    n, d = w.batch * w.num_tables, w.dim
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(w.seed)
    x = torch.randn((n, d), device=dev, generator=g) * 0.05
    q = torch.empty((n, d), dtype=torch.int8, device=dev)
    s = torch.empty(n, dtype=torch.float32, device=dev)
    y = torch.empty((n, d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        E.quantize_rows(x, q, s)
        E.dequantize_rows(q, s, y)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    t_enc = t_dec = 0.0
    for _ in range(args.steps):
        ev[0].record(stream)
        E.quantize_rows(x, q, s)
        ev[1].record(stream)
        E.dequantize_rows(q, s, y)
        ev[2].record(stream)
        torch.cuda.synchronize()
        t_enc += ev[0].elapsed_time(ev[1])
        t_dec += ev[1].elapsed_time(ev[2])
    clk = clocks.stop()
    peak, peak_kind = measured_peaks()
    row_bytes = 4 * d + d + 4  # either direction: fp32 row one way, codes and scale the other
    enc_ms, dec_ms = t_enc / args.steps, t_dec / args.steps
    enc_gbps = n * row_bytes / (enc_ms / 1e3) / 1e9
    dec_gbps = n * row_bytes / (dec_ms / 1e3) / 1e9
    dom, dom_ms, dom_gbps = ("encode", enc_ms, enc_gbps) if enc_ms >= dec_ms else ("decode", dec_ms, dec_gbps)
    S = min(n, 200_000)
    xs = x[:S].cpu().numpy()
    t0 = time.perf_counter()
    import oracle
    qs, ss = oracle.quantize_rows(xs)
    oracle.dequantize_rows(qs, ss)
    cpu_s = time.perf_counter() - t0
    line = {
        "metric": "int8 row codec rows/s (encode + decode)",
        "value": n / ((enc_ms + dec_ms) / 1e3), "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": enc_ms + dec_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32->s8",
        "data": "synthetic",
        "config": {"workload": f"pooled rows of {w.name}: {n} rows x {d} fp32",
                   "l2": f"not flushed: {n * d * 4 / 1e6:.0f} MB of fp32 rows per call"},
        "kernels": {"encode": {"ms_per_launch": enc_ms, "gbps": enc_gbps},
                    "decode": {"ms_per_launch": dec_ms, "gbps": dec_gbps}},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": dom_gbps, "peak": peak,
                     "unit": "GB/s", "frac": dom_gbps / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": n * row_bytes, "ms_per_launch": dom_ms,
                     "peak_kind": peak_kind},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "cpu_baseline": {"value": S / cpu_s, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {S} rows, encode + decode"},
    }
    print(json.dumps(line), flush=True)


def run_cross(args):
    """One cross layer over the concatenated dense and pooled vectors of a batch (one GPU):
    forward and backward timed with CUDA events; the oracle timed on a sample."""
    import time
    import torch
    import recommender_model_embedding_gb300 as E
    w_ = workload(args.small, args.rows_div, args.config, args.batch)
    B, K = w_.batch, (w_.num_tables + 1) * w_.dim
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(w_.seed)
    r = lambda *s: torch.randn(s, device=dev, generator=g)
    x0, xl, dout = r(B, K), r(B, K), r(B, K)
    w, b = r(K) / K ** 0.5, r(K)
    out, dx0, dxl = (torch.empty((B, K), device=dev) for _ in range(3))
    dw, db = torch.empty(K, device=dev), torch.empty(K, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        E.cross_forward(x0, xl, w, b, out)
        E.cross_backward(x0, xl, w, dout, dx0, dxl, dw, db)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    t_f = t_b = 0.0
    for _ in range(args.steps):
        ev[0].record(stream)
        E.cross_forward(x0, xl, w, b, out)
        ev[1].record(stream)
        E.cross_backward(x0, xl, w, dout, dx0, dxl, dw, db)
        ev[2].record(stream)
        torch.cuda.synchronize()
        t_f += ev[0].elapsed_time(ev[1])
        t_b += ev[1].elapsed_time(ev[2])
    clk = clocks.stop()
    peak, peak_kind = measured_peaks()
    f_ms, b_ms = t_f / args.steps, t_b / args.steps
    f_bytes, b_bytes = B * K * 12, B * K * 20  # per sample: 3 rows / 5 rows of K floats
    f_gbps, b_gbps = f_bytes / (f_ms / 1e3) / 1e9, b_bytes / (b_ms / 1e3) / 1e9
    dom = ("backward", b_ms, b_gbps, b_bytes) if b_ms >= f_ms else ("forward", f_ms, f_gbps, f_bytes)
    import oracle
    S = min(B, 256)
    c = lambda a: a[:S].cpu().numpy()
    t0 = time.perf_counter()
    oracle.cross_forward(c(x0), c(xl), w.cpu().numpy(), b.cpu().numpy())
    oracle.cross_backward(c(x0), c(xl), w.cpu().numpy(), c(dout))
    cpu_s = time.perf_counter() - t0
    line = {
        "metric": "cross interaction samples/s (forward + backward)",
        "value": B / ((f_ms + b_ms) / 1e3), "unit": "samples/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": f_ms + b_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"cross layer over {w_.name}: {B} samples x {K} features",
                   "l2": f"not flushed: {B * K * 4 / 1e6:.0f} MB per input tensor"},
        "kernels": {"forward": {"ms_per_launch": f_ms, "gbps": f_gbps},
                    "backward": {"ms_per_launch": b_ms, "gbps": b_gbps}},
        "roofline": {"bound": "hbm", "kernel": dom[0], "achieved": dom[2], "peak": peak,
                     "unit": "GB/s", "frac": dom[2] / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": dom[3], "ms_per_launch": dom[1],
                     "peak_kind": peak_kind},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "cpu_baseline": {"value": S / cpu_s, "unit": "samples/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {S} samples, forward + backward"},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.cross:
        run_cross(args)
    elif args.codec:
        run_codec(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
