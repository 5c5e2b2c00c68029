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
    ap.add_argument("--steps", type=int, default=20)
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
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def workload(small: bool, rows_div: int = 1):
    import dataclasses
    import synth
    w = synth.workload(2, "small" if small else "full")
    if rows_div > 1:
        w = dataclasses.replace(w, rows=[max(100, r // rows_div) for r in w.rows],
                                name=f"{w.name}-rows-div{rows_div}")
    return w


# ------------------------------------------------------------------ CPU oracle timing

def time_oracle(w, batches, seconds: float, sample: int, min_steps: int = 1, max_steps: int = 10**9):
    """Run the oracle's full step on the first `sample` samples of successive batches until
    `seconds` of CPU time have passed (at least min_steps).  Returns (samples/s, steps, s)."""
    import oracle
    import synth
    orc = oracle.Model.from_workload(w)
    T, D = w.num_tables, w.dim
    done, t_total, k = 0, 0.0, 0
    while (t_total < seconds or k < min_steps) and k < max_steps:
        b = batches[k % len(batches)]
        S = min(sample, b.batch)
        ids = b.ids[: S * T]
        dense, dout = b.dense[:S], b.dout[:S]
        t0 = time.perf_counter()
        pooled, _, _ = orc.forward(ids, None, S)
        oracle.interact(dense, pooled, T, D)
        _, dp, _, mp = oracle.interact_backward(dout, dense, pooled, T, D)
        orc.backward_adagrad(dp, mp)
        t_total += time.perf_counter() - t0
        done += S
        k += 1
    return (done / t_total if t_total > 0 else 0.0), k, t_total


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import synth
    w = workload(args.small, args.rows_div)
    batches = [synth.make_batch(w, s) for s in range(min(NUM_BATCHES, args.steps + args.warmup))]
    S = min(args.cpu_sample, w.batch)
    time_oracle(w, batches, 0.0, S, min_steps=args.warmup, max_steps=args.warmup)
    v, k, secs = time_oracle(w, batches, 0.0, S, min_steps=args.steps, max_steps=args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(k, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "global_batch": w.batch, "tables": w.num_tables,
                   "dim": w.dim, "rows_total": int(sum(w.rows)),
                   "ids": "zipf(1.05) over a seeded permutation of ranks", "parallelism": "none"},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"first {S} samples of each {w.batch}-sample batch, full step"},
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


# ------------------------------------------------------------------ algorithmic bytes

def kernel_bytes(w, U: int):
    """Algorithmic bytes of one launch of each step kernel (fp32 tables, one-hot)."""
    B, T, D = w.batch, w.num_tables, w.dim
    Wd = w.out_width
    row = 4 * D
    return {
        # ids read, row/slot written; dedup-set traffic stays in L2
        "map_dedup": B * T * (8 + 4 + 4) + U * 12,
        # gathered rows + dense in, interaction out, per-lookup indices
        "fused_fwd": B * (T * row + row + 4 * Wd) + B * T * 16,
        # re-gathered rows, dense, dout in; d_dense out; per-unique gradient rows written once
        "fused_bwd": B * (T * row + 2 * row + 4 * Wd) + B * T * 4 + U * row,
        # per unique row: g read + zeroed, w and acc read + written
        "adagrad_from_g": U * (6 * row + 8),
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

    w = workload(args.small, args.rows_div)
    B, T, D = w.batch, w.num_tables, w.dim
    Wd = w.out_width
    host_batches = [synth.make_batch(w, s) for s in range(NUM_BATCHES)]
    batches = []
    for hb in host_batches:
        batches.append(dict(ids=torch.from_numpy(hb.ids).to(dev),
                            dense=torch.from_numpy(hb.dense).to(dev),
                            dout=torch.from_numpy(hb.dout).to(dev)))
    out = torch.empty((B, Wd), device=dev)
    ddense = torch.empty((B, D), device=dev)
    ctx = E.EmbCtx.from_workload(w, max_batch=B, max_lookups=B * T)
    stream = torch.cuda.current_stream()

    def step(k):
        bt = batches[k % NUM_BATCHES]
        ctx.forward_interact(bt["ids"], None, B, bt["dense"], out)
        ctx.backward_interact_adagrad(bt["dout"], bt["dense"], ddense)

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
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = ctx.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for k in range(args.steps):
        step(k)
    ev1.record(stream)
    torch.cuda.synchronize()
    launches = ctx.launch_count() - n0
    ms = ev0.elapsed_time(ev1)
    if ws > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
        dist.barrier()
    clk = clocks.stop() if clocks else None
    prof = ctx.profile_read()
    ctx.profile(False)
    keys, _ = ctx.read_unique()
    U = int(keys.size)

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        hb = host_batches[0]
        pin = lambda a: torch.from_numpy(a).pin_memory()
        h_ids, h_dense, h_dout = pin(hb.ids), pin(hb.dense), pin(hb.dout)
        h_out = torch.empty((B, Wd)).pin_memory()
        h_dd = torch.empty((B, D)).pin_memory()
        for _ in range(2):
            ctx.train_step_host(h_ids, None, B, h_dense, h_dout, h_out, h_dd)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            ctx.train_step_host(h_ids, None, B, h_dense, h_dout, h_out, h_dd)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = e0.elapsed_time(e1)
        if ws > 1:
            t = torch.tensor([ems], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ems = float(t.item())
        e2e = {"value": ws * B * args.e2e_steps / (ems / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(h_ids.numel() * 8 + h_dense.numel() * 4 + h_dout.numel() * 4),
               "d2h_bytes_per_step": int(h_out.numel() * 4 + h_dd.numel() * 4),
               "ms_per_step": ems / args.e2e_steps}

    flags = ctx.get_status()
    if rank != 0:
        ctx.close()
        if ws > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    kb = kernel_bytes(w, U)
    per_kernel = {n: {"ms_per_launch": t / c, "launches": c} for n, (t, c) in prof.items()}
    dom = max((n for n in prof if n in kb), key=lambda n: prof[n][0])
    dom_ms = prof[dom][0] / prof[dom][1]
    achieved = kb[dom] / (dom_ms / 1e3) / 1e9
    traffic = traffic_for(dom)
    gathered = B * T * 4 * D
    updated = U * (2 * 4 * D + 2 * 4 * D)
    step_s = ms / args.steps / 1e3
    line = {
        "metric": METRIC,
        "value": ws * B * args.steps / (ms / 1e3),
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
        "config": {"workload": w.name, "global_batch": ws * B, "per_gpu_batch": B,
                   "tables": T, "dim": D, "rows_total": int(sum(w.rows)),
                   "ids": "zipf(1.05) over a seeded permutation of ranks, one per (sample, table)",
                   "interaction": f"{w.num_features} vectors -> {w.num_pairs} pairs + {D} dense",
                   "optimizer": "adagrad per element, lr 0.01, eps 1e-8, acc0 0.1",
                   "l2": ("not flushed: inputs larger than L2 (3 rotating batches, "
                          f"{(B * T * 8 + B * D * 4 + B * Wd * 4) / 1e6:.0f} MB of step inputs and "
                          f"{gathered / 1e6:.0f} MB of gathered rows per step)"),
                   "parallelism": "replicas" if ws > 1 else "single"},
        "headline": {"bytes_per_step": gathered + updated, "gathered_bytes": gathered,
                     "updated_bytes": updated, "unique_rows": U,
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
        "e2e": e2e,
        "device_flags": flags,
    }
    if not args.no_cpu_baseline:
        S = min(args.cpu_sample, B)
        v, k, secs = time_oracle(w, host_batches, args.cpu_seconds, S)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"first {S} samples of the {B}-sample batches, full step, "
                                          f"{k} steps in {secs:.1f} s"}
    print(json.dumps(line), flush=True)
    ctx.close()
    if ws > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
