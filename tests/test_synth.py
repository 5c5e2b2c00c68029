"""The seeded input generators: determinism, shapes and distributions."""
import numpy as np

import synth


def test_batches_are_deterministic_and_steps_differ():
    w = synth.workload(3, "small")
    a, b, c = synth.make_batch(w, 0), synth.make_batch(w, 0), synth.make_batch(w, 1)
    assert np.array_equal(a.ids, b.ids) and np.array_equal(a.offsets, b.offsets)
    assert np.array_equal(a.dout, b.dout)
    assert not np.array_equal(a.ids[:100], c.ids[:100])


def test_shapes_of_every_workload():
    for k in (1, 2, 3, 4, 5):
        w = synth.workload(k, "small")
        b = synth.make_batch(w, 0)
        B, T, D = w.batch, w.num_tables, w.dim
        if w.multi_hot:
            assert b.offsets.shape == (B * T + 1,) and b.offsets[0] == 0 and b.offsets[-1] == b.nnz
            assert b.offsets.dtype == np.int32 and np.all(np.diff(b.offsets) >= 1)
        else:
            assert b.offsets is None and b.nnz == B * T
        if w.interaction:
            assert b.dense.shape == (B, D) and b.dout.shape == (B, D + (T + 1) * T // 2)
        else:
            assert b.dout.shape == (B, T, D)


def test_ids_stay_in_their_tables():
    for k in (1, 2, 3, 5):
        w = synth.workload(k, "small")
        b = synth.make_batch(w, 0)
        lens = np.diff(b.offsets) if b.offsets is not None else np.ones(b.nnz, np.int64)
        table = np.repeat(np.arange(w.batch * w.num_tables) % w.num_tables, lens)
        assert np.all(b.ids >= 0) and np.all(b.ids < np.asarray(w.rows)[table])


def test_criteo_row_counts():
    rows = synth.criteo_rows()
    assert len(rows) == 26 and rows[:8] == [10_000_000] * 8
    assert rows[8] == 100 and rows[-1] == 1_000_000 and sum(rows) == 82_390_542


def test_zipf_sampler_matches_pmf():
    rng = np.random.default_rng(2)
    for n, a in ((1, 1.1), (2, 1.05), (40, 1.1), (1000, 1.05)):
        r = synth.zipf_ranks(rng, n, a, 400_000)
        assert r.min() >= 1 and r.max() <= n
        p = np.arange(1, n + 1, dtype=np.float64) ** -a
        p /= p.sum()
        emp = np.bincount(r, minlength=n + 1)[1:] / r.size
        z = np.abs(emp - p) / np.sqrt(p * (1 - p) / r.size + 1e-300)
        assert z.max() < 5.5


def test_zipf_unique_count_near_expectation():
    w = synth.workload(2)
    rng = np.random.default_rng(5)
    r = synth.zipf_ranks(rng, 1_000_000, 1.05, 65536)
    exp = synth.zipf_expected_unique(1_000_000, 1.05, 65536)
    assert abs(np.unique(r).size - exp) < 0.02 * exp
    assert w.batch == 65536 and w.num_tables == 26 and w.dim == 128


def test_poisson_bag_lengths():
    w = synth.workload(3)
    L = synth.bag_lengths(w, 0)
    assert L.min() >= 1 and L.max() <= 100
    assert abs(L.mean() - 20.0) < 0.05


def test_key_bijection_distinct_nonnegative():
    ranks = np.arange(2_000_000, dtype=np.int64)
    keys = synth.key_bijection(ranks, 123)
    assert keys.min() >= 0 and np.unique(keys).size == ranks.size
