"""GPU edge cases: empty and ragged batches, rejected IDs and keys, malformed offsets, a full
hash table, a duplicate storm on new keys, call-order errors and the host-buffer step."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close, read_gpu_rows, to_dev

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


def _static(E, rows=(50, 70, 30), dim=16, **kw):
    return E.EmbCtx(len(rows), dim, rows=list(rows), seed=99, max_batch=64, max_lookups=512, **kw)


def test_empty_batch(E, torch):
    with _static(E) as ctx:
        ids = torch.empty(0, dtype=torch.int64, device="cuda")
        pooled = torch.empty((0, 3, 16), device="cuda")
        ctx.forward(ids, None, 0, pooled)
        ctx.backward_adagrad(torch.empty((0, 3, 16), device="cuda"))
        assert ctx.get_status() == 0
        assert ctx.read_unique()[0].size == 0
        out = torch.empty((0, ctx.out_width), device="cuda")
        ctx.forward_interact(ids, None, 0, torch.empty((0, 16), device="cuda"), out)
        ctx.backward_interact_adagrad(torch.empty((0, ctx.out_width), device="cuda"),
                                      torch.empty((0, 16), device="cuda"),
                                      torch.empty((0, 16), device="cuda"))
        assert ctx.get_status() == 0


def test_out_of_range_ids_flag_and_add_zero(E, torch):
    orc = oracle.Model(3, 16, rows=[50, 70, 30], seed=99)
    ids = np.array([5, 70, 3, -1, 2, 29, 49, 69, 30], np.int64)
    with _static(E) as ctx:
        pooled = torch.empty((3, 3, 16), device="cuda")
        ctx.forward(to_dev(ids, torch), None, 3, pooled)
        pref, pmag, flags = orc.forward(ids, None, 3)
        assert flags == E.FLAG_ID_RANGE
        assert ctx.get_status() == E.FLAG_ID_RANGE
        assert ctx.get_status() == 0  # cleared by the read
        assert_close(pooled.cpu().numpy(), pref, pmag, 1e-5)
        gk, gc = ctx.read_unique()
        ok, oc = orc.unique()
        np.testing.assert_array_equal(np.sort(gk), ok.astype(np.int64))
        grad = np.random.default_rng(1).standard_normal((3, 3, 16)).astype(np.float32)
        ctx.backward_adagrad(to_dev(grad, torch))
        orc.backward_adagrad(grad.astype(np.float64))
        gw, ga = read_gpu_rows(ctx, orc.base, ok.astype(np.int64))
        rw, ra, mw, ma, _ = orc.read_rows(ok)
        assert_close(gw, rw, mw, 1e-5)
        assert_close(ga, ra, ma, 1e-5)


@pytest.mark.parametrize("offs", [[0, 3, 2, 5, 6, 8, 9], [0, 1, 2, 3, 4, 5, 400], [0, 1, 2, 3, 4, 5, 100000],
                                  [-4, 1, 2, 3, 4, 5, 9]])
def test_malformed_offsets_are_flagged(E, torch, offs):
    ids = np.arange(9, dtype=np.int64) % 30
    with _static(E, pooling=E.POOL_MEAN) as ctx:
        pooled = torch.empty((2, 3, 16), device="cuda")
        ctx.forward(to_dev(ids, torch), to_dev(np.array(offs, np.int32), torch), 2, pooled)
        assert ctx.get_status() & E.FLAG_BAD_OFFSETS
        assert torch.isfinite(pooled).all()


def test_mean_pool_empty_bags_give_zero(E, torch):
    w = synth.Workload("t", batch=5, num_tables=2, dim=8, rows=[40, 40], pooling="mean", seed=3)
    orc = oracle.Model.from_workload(w)
    lens = np.array([0, 3, 2, 0, 1, 4, 0, 0, 5, 1])
    offs = np.concatenate(([0], np.cumsum(lens))).astype(np.int32)
    ids = np.random.default_rng(0).integers(0, 40, size=int(lens.sum())).astype(np.int64)
    with E.EmbCtx.from_workload(w, max_lookups=64) as ctx:
        pooled = torch.empty((5, 2, 8), device="cuda")
        ctx.forward(to_dev(ids, torch), to_dev(offs, torch), 5, pooled)
        pref, pmag, _ = orc.forward(ids, offs, 5)
        p = pooled.cpu().numpy()
        assert np.all(p.reshape(10, 8)[lens == 0] == 0)
        assert_close(p, pref, pmag, 1e-5)


def test_hashed_negative_key_and_full_table(E, torch):
    with E.EmbCtx(1, 8, hashed=True, capacity=1024, max_batch=2048, max_lookups=2048) as ctx:
        keys = np.arange(2000, dtype=np.int64) * 7919 + 11
        keys[5] = -3
        pooled = torch.empty((2000, 1, 8), device="cuda")
        ctx.forward(to_dev(keys, torch), None, 2000, pooled)
        f = ctx.get_status()
        assert f & E.FLAG_TABLE_FULL and f & E.FLAG_BAD_KEY
        k, _, _ = ctx.export_hash()
        assert k.size == 1024 and np.unique(k).size == 1024
        assert np.all(np.isin(k, keys[keys >= 0]))
        assert torch.all(pooled == 0)  # every inserted key starts at 0, failed ones add 0


def test_duplicate_storm_on_new_keys(E, torch):
    """32768 lookups over the same 10 new keys: exactly 10 slots, one per key, and each key
    takes one update with the summed gradient."""
    B = 32768
    keys = (np.arange(B, dtype=np.int64) % 10) * 1_000_003 + 17
    grad = np.random.default_rng(2).standard_normal((B, 1, 8)).astype(np.float32)
    orc = oracle.Model(1, 8, hashed=True, capacity=1 << 12, seed=1)
    with E.EmbCtx(1, 8, hashed=True, capacity=1 << 12, max_batch=B, max_lookups=B) as ctx:
        pooled = torch.empty((B, 1, 8), device="cuda")
        ctx.forward(to_dev(keys, torch), None, B, pooled)
        orc.forward(keys, None, B)
        gk, gc = ctx.read_unique()
        assert gk.size == 10 and np.unique(gk).size == 10
        ok, oc = orc.unique()
        np.testing.assert_array_equal(gk[np.argsort(gk)], ok.astype(np.int64))
        np.testing.assert_array_equal(gc[np.argsort(gk)], oc)
        ctx.backward_adagrad(to_dev(grad, torch))
        orc.backward_adagrad(grad.astype(np.float64))
        k, w, a = ctx.export_hash()
        assert k.size == 10 and np.unique(k).size == 10
        order = np.argsort(k)
        ok, ow, oa = orc.export()
        np.testing.assert_array_equal(k[order], ok.astype(np.int64))
        _, _, mw, ma, _ = orc.read_rows(ok)
        assert_close(w[order], ow, mw, 1e-5)
        assert_close(a[order], oa, ma, 1e-5)


def test_call_order_errors(E, torch):
    with _static(E) as ctx:
        with pytest.raises(E.EmbError) as ei:
            ctx.backward_adagrad(torch.zeros((1, 3, 16), device="cuda"))
        assert ei.value.status == E.EMB_ESTATE
        ids = torch.zeros(3, dtype=torch.int64, device="cuda")
        ctx.forward(ids, None, 1, torch.empty((1, 3, 16), device="cuda"))
        with pytest.raises(E.EmbError) as ei:  # the fused backward needs the fused forward
            ctx.backward_interact_adagrad(torch.zeros((1, ctx.out_width), device="cuda"),
                                          torch.zeros((1, 16), device="cuda"),
                                          torch.empty((1, 16), device="cuda"))
        assert ei.value.status == E.EMB_ESTATE
        ctx.backward_adagrad(torch.zeros((1, 3, 16), device="cuda"))
        with pytest.raises(E.EmbError):  # batch above max_batch
            ctx.forward(torch.zeros(65 * 3, dtype=torch.int64, device="cuda"), None, 65,
                        torch.empty((65, 3, 16), device="cuda"))


def test_forward_twice_without_backward(E, torch):
    """A forward without a backward (inference) leaves the dedup set clean for the next."""
    w = synth.workload(2, "small")
    orc = oracle.Model.from_workload(w)
    with E.EmbCtx.from_workload(w) as ctx:
        for step in range(3):
            b = synth.make_batch(w, step)
            pooled = torch.empty((b.batch, 26, 128), device="cuda")
            ctx.forward(to_dev(b.ids, torch), None, b.batch, pooled)
            orc.forward(b.ids, None, b.batch)
            gk, gc = ctx.read_unique()
            ok, oc = orc.unique()
            np.testing.assert_array_equal(np.sort(gk), ok.astype(np.int64))


def test_interact_forward_twice_then_step(E, torch, monkeypatch):
    """Interaction forwards without a backward, on steps that mark rows looked up more than
    once in the dedup set, leave the set clean: the next full step matches the oracle."""
    from test_parity_gpu import run_fused_step
    monkeypatch.setenv("EMB_ONCE_DIRECT", "1")
    w = synth.workload(2, "small")
    rng = np.random.default_rng(3)
    orc = oracle.Model.from_workload(w)
    with E.EmbCtx.from_workload(w) as ctx:
        for step in range(2):
            b = synth.make_batch(w, step)
            out = torch.empty((b.batch, w.out_width), device="cuda")
            ctx.forward_interact(to_dev(b.ids, torch), None, b.batch, to_dev(b.dense, torch), out)
        run_fused_step(E, torch, ctx, orc, w, synth.make_batch(w, 2), rng)


@pytest.mark.parametrize("once", ["0", "1"])
@pytest.mark.parametrize("batch", [1, 7, 1000])
def test_host_buffer_step_matches_device_step(E, torch, batch, once, monkeypatch):
    """The host-buffer step (copies overlapped with the kernels; for this shape pipelined
    over sample chunks, including ragged last chunks) gives the device step's results, with
    and without the once-row update."""
    monkeypatch.setenv("EMB_ONCE_DIRECT", once)
    w = dataclasses.replace(synth.workload(2, "small"), batch=batch)
    b = synth.make_batch(w, 0)
    B = b.batch
    with E.EmbCtx.from_workload(w) as a, E.EmbCtx.from_workload(w) as h:
        out_d = torch.empty((B, w.out_width), device="cuda")
        dd_d = torch.empty((B, w.dim), device="cuda")
        dense, dout = to_dev(b.dense, torch), to_dev(b.dout, torch)
        a.forward_interact(to_dev(b.ids, torch), None, B, dense, out_d)
        a.backward_interact_adagrad(dout, dense, dd_d)
        pin = lambda x: torch.from_numpy(x).pin_memory()
        out_h = torch.empty((B, w.out_width)).pin_memory()
        dd_h = torch.empty((B, w.dim)).pin_memory()
        h.train_step_host(pin(b.ids), None, B, pin(b.dense), pin(b.dout), out_h, dd_h)
        torch.cuda.synchronize()
        assert torch.equal(out_h, out_d.cpu()) and torch.equal(dd_h, dd_d.cpu())
        # both contexts against the oracle (the gradient sums use atomics, so the two GPU
        # results may differ in the last bits)
        orc = oracle.Model.from_workload(w)
        pref, pmag, _ = orc.forward(b.ids, None, B)
        _, dpr, _, mdp = oracle.interact_backward(b.dout, b.dense, pref, w.num_tables, w.dim, pmag)
        orc.backward_adagrad(dpr, mdp)
        keys, _ = orc.unique()
        rw, ra, mw, ma, _ = orc.read_rows(keys)
        for ctx in (a, h):
            gw, ga = read_gpu_rows(ctx, orc.base, keys.astype(np.int64))
            assert_close(gw, rw, mw, 1e-5, "w")
            assert_close(ga, ra, ma, 1e-5, "acc")


def test_profiling_counts_launches(E, torch):
    w = synth.workload(1)
    b = synth.make_batch(w, 0)
    with E.EmbCtx.from_workload(w) as ctx:
        ctx.profile(True)
        n0 = ctx.launch_count()
        out = torch.empty((w.batch, w.out_width), device="cuda")
        dense = to_dev(b.dense, torch)
        ctx.forward_interact(to_dev(b.ids, torch), to_dev(b.offsets, torch), w.batch, dense, out)
        ctx.backward_interact_adagrad(to_dev(b.dout, torch), dense,
                                      torch.empty((w.batch, w.dim), device="cuda"))
        prof = ctx.profile_read()
        assert set(prof) >= {"map_dedup", "fused_fwd", "fused_bwd", "adagrad_from_g"}
        assert sum(n for _, n in prof.values()) == ctx.launch_count() - n0
        assert all(ms > 0 for ms, _ in prof.values())


@pytest.mark.parametrize("once", ["0", "1"])
def test_bounded_wait_gives_up_and_context_stays_usable(E, torch, once, monkeypatch):
    """The give-up path of a bounded in-kernel wait, without a GPU fault: the test knob sets
    the tensor-core backward's first wait (for the tensor core) to zero polls, so it gives up
    at once.  The kernel must raise EMB_FLAG_WAIT_LIMIT, wait at the full limit for what it
    has in flight and leave; afterwards the GPU and a new context compute a correct step."""
    w = synth.workload(2, "small")
    b = synth.make_batch(w, 0)
    B = b.batch
    monkeypatch.setenv("EMB_FUSED_BWD", "tc")
    monkeypatch.setenv("EMB_ONCE_DIRECT", once)
    monkeypatch.setenv("EMB_WAIT_POLLS", "0")
    with E.EmbCtx.from_workload(w) as ctx:
        dense, dout = to_dev(b.dense, torch), to_dev(b.dout, torch)
        out = torch.empty((B, w.out_width), device="cuda")
        ctx.forward_interact(to_dev(b.ids, torch), None, B, dense, out)
        ctx.backward_interact_adagrad(dout, dense, torch.empty((B, w.dim), device="cuda"))
        assert ctx.get_status() & E.FLAG_WAIT_LIMIT
    monkeypatch.delenv("EMB_WAIT_POLLS")
    from test_parity_gpu import run_fused_step
    with E.EmbCtx.from_workload(w) as ctx:
        orc = oracle.Model.from_workload(w)
        run_fused_step(E, torch, ctx, orc, w, b, np.random.default_rng(3))
