"""The replica (N > 1) path of bench.py on CPU: two gloo ranks rendezvous on 127.0.0.1 as
the torch.distributed launcher sets them up; the timed region's length is the maximum over
the ranks, the rate counts every rank's units over that time, and only rank 0 prints the
reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method="env://")
    assert bench.dist_env() == (ws, rank, rank)
    bench.sync_ranks(ws)
    ms = bench.max_over_ranks(10.0 * (rank + 1), ws, torch.device("cpu"))
    rate = bench.whole_job_rate(1000, ws, 5, ms)
    bench.sync_ranks(ws)
    dist.destroy_process_group()
    q.put((rank, ms, rate))


def test_max_over_ranks_and_rate_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slower rank's 20 ms; 2 ranks x 1000 units x 5 steps in 20 ms
    assert [g[1] for g in got] == [20.0, 20.0]
    assert got[0][2] == pytest.approx(2 * 1000 * 5 / 0.020)
    assert got[0][2] == got[1][2]


def test_single_rank_helpers_are_local():
    sys.path.insert(0, ROOT)
    import bench
    bench.sync_ranks(1)
    assert bench.max_over_ranks(7.5, 1, None) == 7.5
    assert bench.whole_job_rate(65536, 1, 20, 1000.0) == pytest.approx(65536 * 20)


def _reference(rank: int, ws: int):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1")
    return subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--small",
         "--steps", "1", "--warmup", "1", "--cpu-sample", "32", "--gpus", str(ws)],
        env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_on_rank0_only():
    r0, r1 = _reference(0, 2), _reference(1, 2)
    assert r0.returncode == 0, r0.stderr[-2000:]
    assert r1.returncode == 0, r1.stderr[-2000:]
    assert r1.stdout.strip() == ""
    lines = [l for l in r0.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["unit"] == "samples/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
