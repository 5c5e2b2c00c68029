"""Parity at the full workload sizes, in the launch configuration the benchmark times.

The oracle cannot redo a whole 65536- or 262144-sample interaction in test time, so these
tests compare
  - the unique rows (or keys) of the whole batch and their counts: bit-exact;
  - the forward output of a random subset of samples (the oracle runs on those samples);
  - the updated parameters of every row that only the subset's samples touch in the whole
    batch (its gradient comes from those samples alone, so the oracle run on the subset
    gives its exact expected update);
  - rows no lookup touched: bit-identical to their initial values.
"""
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


def _free(torch):
    import gc
    gc.collect()
    torch.cuda.empty_cache()


def _lookup_rows(w, b, base):
    """Global row of every lookup and its sample (static tables)."""
    T = w.num_tables
    lens = np.diff(b.offsets) if b.offsets is not None else np.ones(b.nnz, np.int64)
    bag = np.repeat(np.arange(b.batch * T), lens)
    return base[bag % T] + b.ids, bag // T


def _subset_batch(w, b, samples):
    """The lookups, dense rows and upstream gradients of the chosen samples only."""
    T = w.num_tables
    if b.offsets is None:
        ids = b.ids.reshape(b.batch, T)[samples].reshape(-1)
        offs = None
    else:
        lens = np.diff(b.offsets).reshape(b.batch, T)[samples]
        starts = b.offsets[:-1].reshape(b.batch, T)[samples]
        ids = np.concatenate([b.ids[s:s + l] for s, l in zip(starts.reshape(-1), lens.reshape(-1))])
        offs = np.concatenate(([0], np.cumsum(lens.reshape(-1)))).astype(np.int32)
    dense = None if b.dense is None else b.dense[samples]
    return synth.Batch(ids=ids, offsets=offs, dense=dense, dout=b.dout[samples], batch=len(samples))


def _hot_rows(uniq, counts, base, T, per_table=3, ntables=4):
    """The `per_table` most looked-up rows of `ntables` tables spread over the T tables
    (first, last and two between), as global rows."""
    t_of = np.searchsorted(base, uniq, side="right") - 1
    out = []
    for t in np.unique(np.linspace(0, T - 1, ntables).round().astype(int)):
        sel = np.nonzero(t_of == t)[0]
        out.extend(uniq[sel[np.argsort(counts[sel], kind="stable")[::-1][:per_table]]].tolist())
    return np.array(out, np.int64)


def _oracle_on_samples(w, b, samples):
    """The oracle's full step (forward, interaction and its backward, Adagrad) on exactly the
    given samples, starting from the initial tables."""
    T, D = w.num_tables, w.dim
    sub = _subset_batch(w, b, samples)
    orc = oracle.Model.from_workload(dataclasses.replace(w, batch=len(samples)))
    pref, pmag, _ = orc.forward(sub.ids, sub.offsets, len(samples))
    if w.interaction:
        _, dpr, _, mdp = oracle.interact_backward(sub.dout, sub.dense, pref, T, D, pmag)
        orc.backward_adagrad(dpr, mdp)
    else:
        g = sub.dout.astype(np.float64)
        orc.backward_adagrad(g, np.abs(g))
    return orc


def _run_static(E, torch, k, nsub=384):
    w = synth.workload(k)
    b = synth.make_batch(w, 0)
    rng = np.random.default_rng(100 + k)
    tol = tol_for(w)
    B, T, D = w.batch, w.num_tables, w.dim
    base = np.concatenate(([0], np.cumsum(w.rows)))
    rows, sample_of = _lookup_rows(w, b, base)
    uniq, counts = np.unique(rows, return_counts=True)
    with E.EmbCtx.from_workload(w) as ctx:
        ids, offs = to_dev(b.ids, torch), to_dev(b.offsets, torch)
        if w.interaction:
            dense, dout = to_dev(b.dense, torch), to_dev(b.dout, torch)
            out = torch.empty((B, w.out_width), device="cuda")
            ctx.forward_interact(ids, offs, B, dense, out)
        else:
            pooled = torch.empty((B, T, D), device="cuda")
            ctx.forward(ids, offs, B, pooled)
        assert ctx.get_status() == 0
        gk, gc = ctx.read_unique()
        order = np.argsort(gk)
        np.testing.assert_array_equal(gk[order], uniq)
        np.testing.assert_array_equal(gc[order].astype(np.int64), counts)

        samples = np.sort(rng.choice(B, size=nsub, replace=False))
        sub = _subset_batch(w, b, samples)
        orc = oracle.Model.from_workload(dataclasses.replace(w, batch=nsub))
        pref, pmag, _ = orc.forward(sub.ids, sub.offsets, nsub)
        if w.interaction:
            oref, omag = oracle.interact(sub.dense, pref, T, D, pmag)
            got = out[torch.from_numpy(samples).cuda()].cpu().numpy()
            assert_close(got, oref, omag, tol, "out (sampled)")
            dd = torch.empty((B, D), device="cuda")
            ctx.backward_interact_adagrad(dout, dense, dd)
            ddr, dpr, mdd, mdp = oracle.interact_backward(sub.dout, sub.dense, pref, T, D, pmag)
            assert_close(dd[torch.from_numpy(samples).cuda()].cpu().numpy(), ddr, mdd, tol,
                         "d_dense (sampled)")
            orc.backward_adagrad(dpr, mdp)
        else:
            got = pooled[torch.from_numpy(samples).cuda()].cpu().numpy()
            assert_close(got, pref, pmag, tol, "pooled (sampled)")
            ctx.backward_adagrad(to_dev(b.dout, torch))
            g = sub.dout.astype(np.float64)
            orc.backward_adagrad(g, np.abs(g))
        assert ctx.get_status() == 0
        # rows whose every lookup in the whole batch lies in the chosen samples
        in_sub = np.isin(sample_of, samples)
        cnt_sub = np.unique(rows[in_sub], return_counts=True)
        full_cnt = dict(zip(uniq.tolist(), counts.tolist()))
        own = np.array([r for r, c in zip(*cnt_sub) if full_cnt[r] == c], np.int64)
        assert own.size > 0
        gw, ga = read_gpu_rows(ctx, base, own)
        rw, ra, mw, ma, _ = orc.read_rows(own.astype(np.uint64))
        assert_close(gw, rw, mw, tol, "updated w (sampled rows)")
        assert_close(ga, ra, ma, tol, "updated acc (sampled rows)")
        # Zipf-hot rows (the heaviest reductions: thousands of lookups, split across chunks
        # or reduced by vector atomics): the oracle runs on exactly the samples that look any
        # of them up, so their expected update is exact
        hot = _hot_rows(uniq, counts, base, T)
        hot_cnt = counts[np.searchsorted(uniq, hot)]
        hot_samples = np.unique(sample_of[np.isin(rows, hot)])
        if w.ids_dist == "zipf":
            assert hot_cnt.max() > 1000, hot_cnt
        print(f"hot rows {hot.tolist()} lookups {hot_cnt.tolist()} over {hot_samples.size} samples")
        orc_hot = _oracle_on_samples(w, b, hot_samples)
        gw, ga = read_gpu_rows(ctx, base, hot)
        rw, ra, mw, ma, _ = orc_hot.read_rows(hot.astype(np.uint64))
        assert_close(gw, rw, mw, tol, "updated w (hot rows)")
        assert_close(ga, ra, ma, tol, "updated acc (hot rows)")
        del orc_hot
        # untouched rows keep their initial bits
        for t in rng.choice(T, size=4, replace=False):
            cand = rng.integers(0, w.rows[t], size=256)
            cand = cand[~np.isin(base[t] + cand, uniq)]
            gw, _, _ = ctx.read_rows(int(t), cand)
            rw, _, _, _, _ = orc.read_rows((base[t] + cand).astype(np.uint64))
            assert np.array_equal(gw.view(np.uint32), rw.view(np.uint32))
    _free(torch)


@pytest.mark.parametrize("k,once", [(2, None), (3, None), (5, None), (2, "1"), (5, "1")])
def test_full_size_static(E, k, once, monkeypatch):
    """once="1": rows looked up once in the batch are updated by the interaction backward
    itself (the automatic choice leaves a context's first step on the gradient buffer)."""
    import torch
    if once is None:
        monkeypatch.delenv("EMB_ONCE_DIRECT", raising=False)
    else:
        monkeypatch.setenv("EMB_ONCE_DIRECT", once)
    _run_static(E, torch, k)


def test_full_size_hashed_steps(E):
    """The hashed workload at full size: every key set and count exact over 20 steps; the
    rows of keys looked up only by a sampled subset of one step match the oracle."""
    import torch
    w = synth.workload(4)
    rng = np.random.default_rng(4)
    B, T, D = w.batch, w.num_tables, w.dim
    seen = set()
    with E.EmbCtx.from_workload(w) as ctx:
        for step in range(w.steps):
            b = synth.make_batch(w, step)
            pooled = torch.empty((B, T, D), device="cuda")
            ctx.forward(to_dev(b.ids, torch), None, B, pooled)
            assert ctx.get_status() == 0
            gk, gc = ctx.read_unique()
            uk, uc = np.unique(b.ids, return_counts=True)
            order = np.argsort(gk)
            np.testing.assert_array_equal(gk[order], uk)
            np.testing.assert_array_equal(gc[order].astype(np.int64), uc)
            new = np.setdiff1d(uk, np.fromiter(seen, np.int64, len(seen)) if seen else np.empty(0, np.int64))
            if step in (0, w.steps - 1):
                # keys first seen now start at 0; take keys used only by a sample subset
                samples = np.sort(rng.choice(B, size=512, replace=False))
                sub_keys = b.ids.reshape(B, T)[samples].reshape(-1)
                k_sub, c_sub = np.unique(sub_keys, return_counts=True)
                full = dict(zip(uk.tolist(), uc.tolist()))
                new_set = set(new.tolist())
                own = np.array([kk for kk, cc in zip(k_sub.tolist(), c_sub.tolist())
                                if full[kk] == cc and kk in new_set], np.int64)
                gw0, _, f0 = ctx.read_rows(0, own)
                assert f0.all() and np.all(gw0 == 0)
            ctx.backward_adagrad(to_dev(b.dout, torch))
            if step in (0, w.steps - 1) and own.size:
                orc = oracle.Model(1, D, hashed=True, capacity=w.capacity, lr=w.lr, eps=w.eps,
                                   init_acc=w.init_acc, seed=w.seed)
                sub_ids = b.ids.reshape(B, T)[samples].reshape(-1)
                orc.forward(sub_ids, None, len(samples) * T)
                g = b.dout[samples].reshape(-1, 1, D).astype(np.float64)
                orc.backward_adagrad(g, np.abs(g))
                gw, ga, f = ctx.read_rows(0, own)
                rw, ra, mw, ma, _ = orc.read_rows(own.astype(np.uint64))
                assert f.all()
                assert_close(gw, rw, mw, 1e-5, "hashed w (sampled new keys)")
                assert_close(ga, ra, ma, 1e-5, "hashed acc (sampled new keys)")
            seen.update(uk.tolist())
            assert ctx.get_status() == 0
        keys, _, _ = ctx.export_hash()
        assert keys.size == len(seen) and set(keys.tolist()) == seen
    _free(torch)
