"""Feature admission and eviction on the hashed table (DeepRec announcement,
"EmbeddingVariable": admission and eviction strategies are named there, not defined; the
reading: a key's row is updated only once its lookup count over all steps reaches the
admission minimum; an eviction between steps removes keys idle for more than N steps or
counted fewer than M times, and their slots start afresh).

Every step is compared with the oracle: the set of keys in the table and each key's lookup
count and last step bit-exactly, the number of keys each eviction removes exactly, and the
rows within the fp32 tolerance."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from helpers import build_lib
    build_lib()
    import recommender_model_embedding_gb300 as E
    return E


def _compare_tables(ctx, orc, tol=1e-5):
    gk, gw, ga = ctx.export_hash()
    ok, ow, oa = orc.export()
    order = np.argsort(gk)
    np.testing.assert_array_equal(gk[order], ok.astype(np.int64))
    _, _, mw, ma, _ = orc.read_rows(ok)
    assert_close(gw[order], ow, mw, tol, "w")
    assert_close(ga[order], oa, ma, tol, "acc")
    gc, gl = ctx.key_stats(ok.astype(np.int64))
    oc, ol = orc.key_stats(ok)
    np.testing.assert_array_equal(gc.astype(np.int64), oc.astype(np.int64))
    np.testing.assert_array_equal(gl.astype(np.int64), ol)
    return ok


# (step after which to evict, max_idle, min_count)
EVICTIONS = {2: (1, 0), 3: (0, 3), 4: (2, 2)}


@pytest.mark.parametrize("admit", [0, 3])
def test_admission_and_eviction_unfused(E, admit):
    import torch
    w = synth.workload(4, "small")
    with E.EmbCtx.from_workload(w) as ctx:
        orc = oracle.Model.from_workload(w)
        ctx.set_admission(admit)
        orc.set_admission(admit)
        for step in range(6):
            b = synth.make_batch(w, step)
            pooled = torch.empty((b.batch, w.num_tables, w.dim), device="cuda")
            ctx.forward(to_dev(b.ids, torch), None, b.batch, pooled)
            pref, pmag, flags = orc.forward(b.ids, None, b.batch)
            assert ctx.get_status() == flags == 0
            assert_close(pooled.cpu().numpy(), pref, pmag, 1e-5, "pooled")
            ctx.backward_adagrad(to_dev(b.dout, torch))
            g = b.dout.astype(np.float64)
            orc.backward_adagrad(g, np.abs(g))
            assert ctx.get_status() == 0
            _compare_tables(ctx, orc)
            if step in EVICTIONS:
                idle, cnt = EVICTIONS[step]
                n_gpu, n_orc = ctx.evict(idle, cnt), orc.evict(idle, cnt)
                assert n_gpu == n_orc and n_orc > 0
                _compare_tables(ctx, orc)


def test_admission_and_eviction_fused_interaction(E):
    """The fused interaction step on a hashed table (generic fused kernels, 8 features)."""
    import torch
    base = synth.workload(4, "small")
    w = dataclasses.replace(base, num_tables=8, interaction=True, batch=257, seed=base.seed + 8)
    with E.EmbCtx.from_workload(w) as ctx:
        orc = oracle.Model.from_workload(w)
        ctx.set_admission(2)
        orc.set_admission(2)
        T, D = w.num_tables, w.dim
        for step in range(5):
            b = synth.make_batch(w, step)
            dense, dout = to_dev(b.dense, torch), to_dev(b.dout, torch)
            out = torch.empty((b.batch, w.out_width), device="cuda")
            ctx.forward_interact(to_dev(b.ids, torch), None, b.batch, dense, out)
            pref, pmag, _ = orc.forward(b.ids, None, b.batch)
            oref, omag = oracle.interact(b.dense, pref, T, D, pmag)
            assert_close(out.cpu().numpy(), oref, omag, 1e-5, "out")
            dd = torch.empty((b.batch, D), device="cuda")
            ctx.backward_interact_adagrad(dout, dense, dd)
            _, dpr, _, mdp = oracle.interact_backward(b.dout, b.dense, pref, T, D, pmag)
            orc.backward_adagrad(dpr, mdp)
            assert ctx.get_status() == 0
            _compare_tables(ctx, orc)
            if step == 2:
                assert ctx.evict(1, 0) == orc.evict(1, 0)
                _compare_tables(ctx, orc)


def test_reinsert_after_eviction_reuses_slots(E):
    """Evicted slots become tombstones that probes pass and inserts reuse: a table of 128
    slots takes 12 batches of 5 recurring and 35 fresh keys (425 keys in all).  After each
    step, keys idle for more than one step are evicted (every fourth step instead: keys
    counted fewer than twice), so the recurring keys stay in chains full of tombstones."""
    import torch
    D, cap = 4, 128
    with E.EmbCtx(1, D, hashed=True, capacity=cap, max_batch=64, max_lookups=64, seed=3) as ctx:
        orc = oracle.Model(1, D, hashed=True, capacity=cap, seed=3)
        ctx.set_admission(0)                         # counts and last steps, no hold
        with pytest.raises(E.EmbError):              # eviction reads them: not before this
            E.EmbCtx(1, D, hashed=True, capacity=cap, seed=3).evict(1, 0)
        rng = np.random.default_rng(9)
        total = 0
        for step in range(12):
            keys = np.concatenate((np.arange(5), rng.integers(5, 1 << 40, size=35))).astype(np.int64)
            pooled = torch.empty((40, 1, D), device="cuda")
            ctx.forward(to_dev(keys, torch), None, 40, pooled)
            pref, pmag, flags = orc.forward(keys, None, 40)
            assert ctx.get_status() == flags == 0
            assert_close(pooled.cpu().numpy(), pref, pmag, 1e-5, "pooled")
            g = rng.standard_normal((40, 1, D)).astype(np.float32)
            ctx.backward_adagrad(to_dev(g, torch))
            orc.backward_adagrad(g.astype(np.float64), np.abs(g.astype(np.float64)))
            _compare_tables(ctx, orc)
            idle, cnt = (0, 2) if step % 4 == 3 else (1, 0)
            n = orc.evict(idle, cnt)
            assert ctx.evict(idle, cnt) == n
            total += n
            _compare_tables(ctx, orc)
        assert total >= 12 * 35 - cap             # most fresh keys went through a tombstone


def test_eviction_on_a_two_slot_table(E):
    """The smallest table (two slots, no whole group of four): both keys evicted by count,
    a new key then inserts into a tombstone."""
    import torch
    with E.EmbCtx(1, 4, hashed=True, capacity=2, max_batch=8, max_lookups=8, seed=1) as ctx:
        orc = oracle.Model(1, 4, hashed=True, capacity=2, seed=1)
        ctx.set_admission(0)
        for keys in ([1, 2], [3]):
            keys = np.array(keys, np.int64)
            pooled = torch.empty((keys.size, 1, 4), device="cuda")
            ctx.forward(to_dev(keys, torch), None, keys.size, pooled)
            _, _, flags = orc.forward(keys, None, keys.size)
            assert ctx.get_status() == flags
            g = np.ones((keys.size, 1, 4))
            ctx.backward_adagrad(to_dev(g.astype(np.float32), torch))
            orc.backward_adagrad(g, g)
            _compare_tables(ctx, orc)
            assert ctx.evict(0, 2) == orc.evict(0, 2)
            _compare_tables(ctx, orc)
