"""Tiered static tables: every row lives in the host tier (host-mapped memory), HBM caches the
rows batches look up, eviction writes rows back.  The results must be those of a plain
static table: every step is checked against the (single-tier) oracle, with evictions between
steps so that rows leave the cache and come back from the host tier."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from helpers import to_dev
from test_parity_gpu import run_fused_step, run_unfused_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from helpers import build_lib
    build_lib()
    import recommender_model_embedding_gb300 as E
    return E


@pytest.fixture(scope="module")
def torch():
    import torch
    return torch


@pytest.mark.parametrize("k,fused,cache", [(2, True, 1 << 16), (5, True, 1 << 18),
                                            (3, False, 1 << 18), (2, False, 1 << 16)])
def test_tiered_steps_match_single_tier(E, torch, k, fused, cache):
    """Criteo-shaped (fused and unfused), uniform (fused, rows looked up once updated in the
    backward) and multi-hot bf16 row-wise (unfused): six steps; after each, keys idle for more
    than one step are evicted (every third step: keys counted fewer than three times)."""
    w = synth.workload(k, "small")
    rng = np.random.default_rng(80 + k)
    with E.EmbCtx.from_workload(w, cache_rows=cache) as ctx:
        orc = oracle.Model.from_workload(w)
        evicted = 0
        for step in range(6):
            b = synth.make_batch(w, step)
            (run_fused_step if fused else run_unfused_step)(E, torch, ctx, orc, w, b, rng)
            idle, cnt = (0, 3) if step % 3 == 2 else (1, 0)
            evicted += ctx.evict(idle, cnt)
        assert evicted > 0


def test_tiered_cache_full_is_flagged(E, torch):
    """A batch with more distinct rows than the cache holds: the rows that find no slot are
    rejected like a full hashed table (flag raised, they add zero); nothing else breaks, and
    the flag stays raised across later steps until it is read."""
    w = synth.workload(2, "small")
    b = synth.make_batch(w, 0)
    with E.EmbCtx.from_workload(w, cache_rows=1 << 10) as ctx:
        pooled = torch.empty((b.batch, w.num_tables, w.dim), device="cuda")
        ctx.forward(to_dev(b.ids, torch), None, b.batch, pooled)
        ctx.backward_adagrad(torch.zeros_like(pooled))
        assert ctx.evict(0, 1 << 30) > 0      # everything back to the host tier
        small = synth.make_batch(dataclasses.replace(w, batch=8), 1)
        pooled = torch.empty((8, w.num_tables, w.dim), device="cuda")
        ctx.forward(to_dev(small.ids, torch), None, 8, pooled)   # fits: raises nothing
        assert ctx.get_status() == E.FLAG_TABLE_FULL              # the first batch's flag
        assert ctx.get_status() == 0                              # cleared by the read
