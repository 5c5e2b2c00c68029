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


def _batch_rows(w, base, b):
    """Distinct global rows of a batch's valid lookups (numpy, from the ids alone)."""
    T = w.num_tables
    ids = np.asarray(b.ids, np.int64)
    if b.offsets is None:
        t = np.arange(ids.size) % T
    else:
        offs = np.asarray(b.offsets, np.int64)
        t = np.repeat(np.arange(offs.size - 1) % T, np.diff(offs))
    rows = np.diff(base)[t]
    ok = (ids >= 0) & (ids < rows)
    return set((base[t[ok]] + ids[ok]).tolist())


@pytest.mark.parametrize("k,fused,cache", [(2, True, 1 << 16), (3, False, 1 << 18)])
def test_tiered_prefetch_on_side_stream(E, torch, k, fused, cache):
    """While each step's forward and backward run, the next batch is prefetched on a second
    stream; evictions (idle > 1 step) come between steps.  Every step matches the oracle, and
    after a prefetch the next forward finds all its rows cached: the cache occupancy does not
    change across that forward."""
    w = synth.workload(k, "small")
    rng = np.random.default_rng(90 + k)
    side = torch.cuda.Stream()
    batches = [synth.make_batch(w, s) for s in range(6)]
    keep = []  # device copies of prefetched ids, alive until their stream has run
    with E.EmbCtx.from_workload(w, cache_rows=cache) as ctx:
        orc = oracle.Model.from_workload(w)
        for s, b in enumerate(batches):
            occ_before = ctx.tier_occupancy()

            def after_forward(s=s, occ_before=occ_before):
                if s > 0:  # the previous prefetch covered this batch
                    assert ctx.tier_occupancy() == occ_before
                if s + 1 < len(batches):
                    nb = batches[s + 1]
                    ids, offs = to_dev(nb.ids, torch), to_dev(nb.offsets, torch)
                    keep.append((ids, offs))
                    side.wait_stream(torch.cuda.current_stream())  # the ids are copied there
                    ctx.prefetch(ids, offs, nb.batch, stream=side)

            (run_fused_step if fused else run_unfused_step)(E, torch, ctx, orc, w, b, rng,
                                                             after_forward)
            ctx.evict(1, 0)
        torch.cuda.synchronize()


@pytest.mark.parametrize("k,fused", [(2, True), (3, False)])
def test_tiered_watermark_keeps_occupancy_exact(E, torch, k, fused):
    """Watermark high = 1, low = 0: after every backward the cache keeps exactly the rows
    the step looked up plus those prefetched for the next step (every other row is idle
    for at least one step and written back).  Every step matches the oracle."""
    w = synth.workload(k, "small")
    rng = np.random.default_rng(95 + k)
    side = torch.cuda.Stream()
    batches = [synth.make_batch(w, s) for s in range(5)]
    keep = []
    with E.EmbCtx.from_workload(w, cache_rows=1 << 18) as ctx:
        orc = oracle.Model.from_workload(w)
        base = orc.base.astype(np.int64)
        ctx.set_tier_watermark(1, 0)
        for s, b in enumerate(batches):
            prefetch = s % 2 == 1 and s + 1 < len(batches)

            def after_forward(s=s, prefetch=prefetch):
                if prefetch:
                    nb = batches[s + 1]
                    ids, offs = to_dev(nb.ids, torch), to_dev(nb.offsets, torch)
                    keep.append((ids, offs))
                    side.wait_stream(torch.cuda.current_stream())
                    ctx.prefetch(ids, offs, nb.batch, stream=side)

            (run_fused_step if fused else run_unfused_step)(E, torch, ctx, orc, w, b, rng,
                                                             after_forward)
            want = _batch_rows(w, base, b)
            if prefetch:
                want |= _batch_rows(w, base, batches[s + 1])
            assert ctx.tier_occupancy() == len(want)


def test_tiered_watermark_band(E, torch):
    """A watermark band wider than one step: occupancy stays at or below `high` after every
    step, the check evicts at some point, and results match the oracle throughout."""
    w = synth.workload(2, "small")
    rng = np.random.default_rng(99)
    batches = [synth.make_batch(w, s) for s in range(6)]
    with E.EmbCtx.from_workload(w, cache_rows=1 << 16) as ctx:
        orc = oracle.Model.from_workload(w)
        base = orc.base.astype(np.int64)
        per_step = max(len(_batch_rows(w, base, b)) for b in batches)
        high, low = int(1.6 * per_step), int(1.2 * per_step)
        ctx.set_tier_watermark(high, low)
        seen, occ = set(), []
        for b in batches:
            run_fused_step(E, torch, ctx, orc, w, b, rng)
            seen |= _batch_rows(w, base, b)
            occ.append(ctx.tier_occupancy())
            assert occ[-1] <= high
        assert len(seen) > high  # without the check the cache would have grown past high
        ctx.set_tier_watermark(0, 0)


def test_tier_calls_reject_static_and_bad_marks(E, torch):
    w = synth.workload(2, "small")
    b = synth.make_batch(w, 0)
    with E.EmbCtx.from_workload(w) as ctx:  # single tier
        ids = to_dev(b.ids, torch)
        for call in (lambda: ctx.set_tier_watermark(10, 5), ctx.tier_occupancy,
                     lambda: ctx.prefetch(ids, None, b.batch)):
            with pytest.raises(E.EmbError) as ei:
                call()
            assert ei.value.status == E.EMB_EINVAL
    with E.EmbCtx.from_workload(w, cache_rows=1 << 12) as ctx:
        for hi, lo in ((10, 10), (10, -1), ((1 << 12) + 1, 0)):
            with pytest.raises(E.EmbError) as ei:
                ctx.set_tier_watermark(hi, lo)
            assert ei.value.status == E.EMB_EINVAL
        ctx.set_tier_watermark(100, 0)
        assert ctx.tier_occupancy() == 0
