"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on the same seeded
inputs.  Integer results (unique rows, counts, hashed keys, status flags) must match
exactly; floats within 1e-5 (fp32 tables) or 2e-2 (bf16 tables) of the oracle, relative to
max(|ref|, magnitude of the expression)."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close, read_gpu_rows, to_dev, tol_for

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


def _check_unique(ctx, orc, hashed):
    gk, gc = ctx.read_unique()
    ok, oc = orc.unique()
    order = np.argsort(gk)
    np.testing.assert_array_equal(gk[order].astype(np.uint64) if not hashed else gk[order],
                                  ok if not hashed else ok.astype(np.int64))
    np.testing.assert_array_equal(gc[order].astype(np.int64), oc)
    return ok


def _check_rows(ctx, orc, w, keys, tol):
    if w.hashed:
        gw, ga, found = ctx.read_rows(0, keys.astype(np.int64))
        assert found.all()
    else:
        gw, ga = read_gpu_rows(ctx, orc.base, keys.astype(np.int64))
    rw, ra, mw, ma, _ = orc.read_rows(keys)
    assert_close(gw, rw, mw, tol, "updated w")
    assert_close(ga, ra, ma, tol, "updated acc")


def _check_untouched(ctx, orc, w, rng, n=64):
    """Rows no step has looked up are still bit-identical to their initial values."""
    if w.hashed:
        return
    touched = orc.export()[0]
    T = w.num_tables
    for _ in range(4):
        t = int(rng.integers(0, T))
        ids = rng.integers(0, w.rows[t], size=n)
        keys = orc.global_rows(t, ids)
        ids = ids[~np.isin(keys, touched)]
        if ids.size == 0:
            continue
        gw, ga, _ = ctx.read_rows(t, ids)
        rw, ra, _, _, _ = orc.read_rows(orc.global_rows(t, ids))
        assert np.array_equal(gw.view(np.uint32), rw.view(np.uint32)), "untouched rows changed"
        assert np.array_equal(ga, ra)


def run_unfused_step(E, torch, ctx, orc, w, b, rng, after_forward=None):
    """One checked step; after_forward() (if given) runs once the forward is enqueued."""
    tol = tol_for(w)
    B, T, D = b.batch, w.num_tables, w.dim
    ids, offs = to_dev(b.ids, torch), to_dev(b.offsets, torch)
    pooled = torch.empty((B, T, D), device="cuda")
    ctx.forward(ids, offs, B, pooled)
    if after_forward:
        after_forward()
    pref, pmag, flags = orc.forward(b.ids, b.offsets, B)
    assert ctx.get_status() == flags
    assert_close(pooled.cpu().numpy(), pref, pmag, tol, "pooled")
    keys = _check_unique(ctx, orc, w.hashed)
    if w.interaction:
        dense = to_dev(b.dense, torch)
        out = torch.empty((B, w.out_width), device="cuda")
        ctx.interact(dense, pooled, B, out)
        oref, omag = oracle.interact(b.dense, pref, T, D, pmag)
        assert_close(out.cpu().numpy(), oref, omag, tol, "interaction out")
        dout = to_dev(b.dout, torch)
        dd = torch.empty((B, D), device="cuda")
        dp = torch.empty((B, T, D), device="cuda")
        ctx.interact_backward(dout, dense, pooled, B, dd, dp)
        ddr, dpr, mdd, mdp = oracle.interact_backward(b.dout, b.dense, pref, T, D, pmag)
        assert_close(dd.cpu().numpy(), ddr, mdd, tol, "d_dense")
        assert_close(dp.cpu().numpy(), dpr, mdp, tol, "d_pooled")
        grad_dev, grad_ref, grad_mag = dp, dpr, mdp
    else:
        grad_dev = to_dev(b.dout, torch)
        grad_ref = b.dout.astype(np.float64)
        grad_mag = np.abs(grad_ref)
    ctx.backward_adagrad(grad_dev)
    assert orc.backward_adagrad(grad_ref, grad_mag) == 0
    assert ctx.get_status() == 0
    _check_rows(ctx, orc, w, keys, tol)
    _check_untouched(ctx, orc, w, rng)


def run_fused_step(E, torch, ctx, orc, w, b, rng, after_forward=None):
    tol = tol_for(w)
    B, T, D = b.batch, w.num_tables, w.dim
    ids, offs = to_dev(b.ids, torch), to_dev(b.offsets, torch)
    dense, dout = to_dev(b.dense, torch), to_dev(b.dout, torch)
    out = torch.empty((B, w.out_width), device="cuda")
    ctx.forward_interact(ids, offs, B, dense, out)
    if after_forward:
        after_forward()
    pref, pmag, flags = orc.forward(b.ids, b.offsets, B)
    oref, omag = oracle.interact(b.dense, pref, T, D, pmag)
    assert ctx.get_status() == flags
    assert_close(out.cpu().numpy(), oref, omag, tol, "fused out")
    keys = _check_unique(ctx, orc, w.hashed)
    dd = torch.empty((B, D), device="cuda")
    ctx.backward_interact_adagrad(dout, dense, dd)
    ddr, dpr, mdd, mdp = oracle.interact_backward(b.dout, b.dense, pref, T, D, pmag)
    assert_close(dd.cpu().numpy(), ddr, mdd, tol, "fused d_dense")
    assert orc.backward_adagrad(dpr, mdp) == 0
    assert ctx.get_status() == 0
    _check_rows(ctx, orc, w, keys, tol)
    _check_untouched(ctx, orc, w, rng)


@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_unfused_path_small(E, torch, k):
    w = synth.workload(k, "small")
    rng = np.random.default_rng(k)
    with E.EmbCtx.from_workload(w) as ctx:
        orc = oracle.Model.from_workload(w)
        for step in range(2):
            run_unfused_step(E, torch, ctx, orc, w, synth.make_batch(w, step), rng)


# fused-kernel choice -> (EMB_FUSED_FWD, EMB_FUSED_BWD, EMB_ONCE_DIRECT)
_IMPLS = {
    "tc-once": ("tc", "tc", "1"),  # rows looked up once updated inside the backward
    "tc-g": ("tc", "tc", "0"),     # every row through the gradient buffer
    "simt": ("simt", "simt", "0"), # FMA-pipe forward and backward
}


@pytest.fixture(params=list(_IMPLS))
def bwd_impl(request, monkeypatch):
    """Fused interaction kernels, chosen when a context is created: the tensor-core forward
    and backward (fp32, one-hot, D = 128) in their variants, or the FMA-pipe kernels."""
    fwd, bwd, once = _IMPLS[request.param]
    monkeypatch.setenv("EMB_FUSED_FWD", fwd)
    monkeypatch.setenv("EMB_FUSED_BWD", bwd)
    monkeypatch.setenv("EMB_ONCE_DIRECT", once)
    return request.param


@pytest.mark.parametrize("k", [1, 2, 5])
def test_fused_path_small(E, torch, k, bwd_impl):
    w = synth.workload(k, "small")
    rng = np.random.default_rng(10 + k)
    with E.EmbCtx.from_workload(w) as ctx:
        orc = oracle.Model.from_workload(w)
        for step in range(2):
            run_fused_step(E, torch, ctx, orc, w, synth.make_batch(w, step), rng)


@pytest.mark.parametrize("T", [7, 20, 26, 31])
@pytest.mark.parametrize("batch", [1, 5, 1000])
def test_fused_feature_counts(E, torch, T, batch, bwd_impl):
    """Interaction vector counts F = T+1 up to the maximum 32 (a full 32 x 32 operand tile),
    with batches below, near and above one sample per CTA; T = 26 runs the kernels compiled
    for F = 27, here also with odd batches (a last pair of one sample)."""
    base = synth.workload(2, "small")
    rows = (base.rows * 2)[:T]
    w = dataclasses.replace(base, num_tables=T, rows=rows, batch=batch, seed=base.seed + T)
    rng = np.random.default_rng(T * 1000 + batch)
    with E.EmbCtx.from_workload(w) as ctx:
        orc = oracle.Model.from_workload(w)
        for step in range(2):
            run_fused_step(E, torch, ctx, orc, w, synth.make_batch(w, step), rng)


def test_hashed_steps_small(E, torch):
    w = synth.workload(4, "small")
    rng = np.random.default_rng(4)
    with E.EmbCtx.from_workload(w) as ctx:
        orc = oracle.Model.from_workload(w)
        for step in range(w.steps):
            run_unfused_step(E, torch, ctx, orc, w, synth.make_batch(w, step), rng)
        gk, gw, ga = ctx.export_hash()
        ok, ow, oa = orc.export()
        order = np.argsort(gk)
        np.testing.assert_array_equal(gk[order], ok.astype(np.int64))
        _, _, mw, ma, _ = orc.read_rows(ok)
        assert_close(gw[order], ow, mw, 1e-5, "exported w")
        assert_close(ga[order], oa, ma, 1e-5, "exported acc")


@pytest.mark.parametrize("once", ["0", "1"])
def test_mixed_fused_and_unfused_steps(E, torch, once, monkeypatch):
    """The two backward paths leave the same state behind (the dedup set included, whose
    values the once-row steps mark): alternate them on one context."""
    monkeypatch.setenv("EMB_ONCE_DIRECT", once)
    w = synth.workload(2, "small")
    rng = np.random.default_rng(7)
    with E.EmbCtx.from_workload(w) as ctx:
        orc = oracle.Model.from_workload(w)
        for step in range(4):
            b = synth.make_batch(w, step)
            (run_fused_step if step % 2 else run_unfused_step)(E, torch, ctx, orc, w, b, rng)


def test_once_rows_automatic_switch(E, torch, monkeypatch):
    """Automatic choice of the once-row update: it follows the previous batch's share of
    unique rows, so steps alternating between a mostly-unique uniform batch and a Zipf batch
    switch it on and off across steps; every step still matches the oracle."""
    monkeypatch.delenv("EMB_ONCE_DIRECT", raising=False)
    monkeypatch.setenv("EMB_FUSED_BWD", "tc")
    wu = synth.workload(5, "small")
    wz = dataclasses.replace(wu, ids_dist="zipf", alpha=1.2)
    rng = np.random.default_rng(55)
    with E.EmbCtx.from_workload(wu) as ctx:
        orc = oracle.Model.from_workload(wu)
        for step, w in enumerate([wu, wu, wu, wz, wz, wu, wz, wu]):
            run_fused_step(E, torch, ctx, orc, w, synth.make_batch(w, step), rng)


@pytest.mark.parametrize("k,fused", [(2, True), (2, False), (3, False), (4, False)])
def test_adagrad_decay_steps(E, torch, k, fused):
    """Adagrad Decay (accumulators discounted by 0.5 per period of two steps) on the fused
    path (Criteo-shaped), the unfused path (multi-hot bf16 row-wise and the hashed table):
    five steps, every one against the oracle."""
    w = synth.workload(k, "small")
    rng = np.random.default_rng(70 + k)
    with E.EmbCtx.from_workload(w) as ctx:
        orc = oracle.Model.from_workload(w)
        ctx.set_adagrad_decay(0.5, 2)
        orc.set_adagrad_decay(0.5, 2)
        for step in range(5):
            b = synth.make_batch(w, step)
            (run_fused_step if fused else run_unfused_step)(E, torch, ctx, orc, w, b, rng)


@pytest.mark.parametrize("k", [1, 3])
def test_multi_hot_and_one_hot_steps(E, torch, k):
    """A multi-hot step leaves its rows' sums in the gradient buffer (the summing reduce
    stores them and the update reads them without clearing); a later step whose reduce adds
    into that buffer (one-hot batches, the fused interaction backward) zeroes what is left
    first.  Alternate the two batch kinds on one context; every step against the oracle."""
    wm = synth.workload(k, "small")
    wo = dataclasses.replace(wm, bag="one")
    rng = np.random.default_rng(90 + k)
    seq = [(wm, run_unfused_step), (wo, run_unfused_step), (wm, run_unfused_step),
           (wm, run_unfused_step)]
    if wm.interaction:
        seq += [(wo, run_fused_step), (wm, run_unfused_step), (wo, run_fused_step)]
    with E.EmbCtx.from_workload(wm) as ctx:
        orc = oracle.Model.from_workload(wm)
        for step, (w, run) in enumerate(seq):
            run(E, torch, ctx, orc, w, synth.make_batch(w, step), rng)


@pytest.mark.parametrize("k,fused", [(2, True), (2, False), (1, False), (1, True)])
def test_rowwise_fp32_steps(E, torch, k, fused):
    """Row-wise Adagrad on fp32 tables: the update kernel that stages its rows in shared
    memory, after the fused interaction backward (one-hot Criteo shape, gradient buffer
    cleared by the update) and after the summing reduce of multi-hot batches (buffer left
    as stored); three steps each against the oracle."""
    w = dataclasses.replace(synth.workload(k, "small"), optimizer="adagrad_row")
    rng = np.random.default_rng(120 + k)
    with E.EmbCtx.from_workload(w) as ctx:
        orc = oracle.Model.from_workload(w)
        for step in range(3):
            b = synth.make_batch(w, step)
            (run_fused_step if fused else run_unfused_step)(E, torch, ctx, orc, w, b, rng)
