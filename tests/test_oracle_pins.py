"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against a hand-derived fixture (tests/golden), a
closed form, a library routine on a special case, finite differences, or brute force in
numpy on tiny inputs.  The pins are chosen so that a dropped term, a wrong sign, a wrong
index or a transposed operand in the oracle fails at least one of them.
"""
import json
import os
from decimal import Decimal

import numpy as np
import pytest

import oracle
import synth


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ generator and storage

def test_splitmix64_reference_vectors(golden_dir):
    g = _golden(golden_dir, "splitmix64_seed0.json")
    got = [oracle.splitmix64(g["seed"], n) for n in (1, 2, 3)]
    assert got == [int(h, 16) for h in g["outputs_hex"]]


def test_init_values_uniform_on_interval():
    # 96k values over a grid of (table, row, column); U(-0.05, 0.05): range, mean, KS.
    vals = np.array([oracle.init_value(0x5EED0002, t, r, c)
                     for t in range(3) for r in range(0, 4000, 5) for c in range(0, 128, 3)],
                    dtype=np.float64)
    assert vals.min() >= -0.05 and vals.max() < 0.05
    assert abs(vals.mean()) < 3 * 0.1 / np.sqrt(12 * vals.size)
    u = np.sort((vals + 0.05) / 0.1)
    ks = np.max(np.abs(u - (np.arange(1, u.size + 1) - 0.5) / u.size))
    assert ks < 1.63 / np.sqrt(u.size)  # 1% level of the Kolmogorov distribution
    # the counter layout gives every (table, row, column) its own stream position: repeated
    # values stay at the birthday-bound level of 24-bit draws (about n^2 / 2^25)
    dups = vals.size - np.unique(vals).size
    assert dups < 2 * vals.size ** 2 / 2 ** 25 + 50


def test_init_values_depend_on_seed_table_row_col():
    base = oracle.init_value(1, 2, 3, 4)
    assert oracle.init_value(2, 2, 3, 4) != base
    assert oracle.init_value(1, 3, 3, 4) != base
    assert oracle.init_value(1, 2, 4, 4) != base
    assert oracle.init_value(1, 2, 3, 5) != base


def test_bf16_round_to_nearest_even_matches_library():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-6, 6, 20000),
        # exact halfway cases: low 16 bits = 0x8000 with even and odd kept bit
        (np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x40490000 | 0x8000], np.uint32)).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 1e-40, 3.0e38], np.float32),
    ])
    ours = np.array([oracle.bf16_rne_bits(x) for x in xs], np.uint16)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


# ------------------------------------------------------------------ pooling

def _tiny_static(mean=False, bf16=False, rows=(50, 70, 30)):
    return oracle.Model(len(rows), 8, rows=list(rows), bf16=bf16, mean=mean, seed=99)


def _dense_tables(m):
    """Every row of every table read back, as plain arrays (the brute force's tables)."""
    tabs = []
    for t in range(m.T):
        w, _, _, _, _ = m.read_rows(m.global_rows(t, np.arange(m.rows[t])))
        tabs.append(w.astype(np.float64))
    return tabs


@pytest.mark.parametrize("mean", [False, True])
def test_pool_matches_brute_force(mean):
    m = _tiny_static(mean=mean)
    tabs = _dense_tables(m)
    rng = np.random.default_rng(3)
    B, T = 9, m.T
    lens = rng.integers(0, 6, size=B * T)
    offs = np.concatenate(([0], np.cumsum(lens))).astype(np.int32)
    ids = np.concatenate([rng.integers(0, m.rows[i % T], size=lens[i]) for i in range(B * T)]).astype(np.int64)
    pooled, mag, flags = m.forward(ids, offs, B)
    assert flags == 0
    for b in range(B):
        for t in range(T):
            bag = b * T + t
            sel = ids[offs[bag]:offs[bag + 1]]
            expect = tabs[t][sel].sum(axis=0) if sel.size else np.zeros(m.D)
            emag = np.abs(tabs[t][sel]).sum(axis=0) if sel.size else np.zeros(m.D)
            if mean and sel.size:
                expect = expect / sel.size
                emag = emag / sel.size
            np.testing.assert_allclose(pooled[b, t], expect, rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(mag[b, t], emag, rtol=1e-13, atol=1e-15)


def test_one_hot_pool_is_the_row_itself():
    m = _tiny_static()
    tabs = _dense_tables(m)
    B = 11
    ids = np.stack([np.arange(B) % m.rows[t] for t in range(m.T)], axis=1).reshape(-1)
    pooled, _, _ = m.forward(ids, None, B)
    for b in range(B):
        for t in range(m.T):
            assert np.array_equal(pooled[b, t].astype(np.float32), tabs[t][ids[b * m.T + t]].astype(np.float32))


def test_out_of_range_ids_flag_and_add_zero():
    m = _tiny_static()
    tabs = _dense_tables(m)
    ids = np.array([5, 70, 3, -1, 2, 29], np.int64)  # bag 1 (t=1) id 70 == rows; bag 3 negative
    pooled, _, flags = m.forward(ids, None, 2)
    assert flags & oracle.FLAG_ID_RANGE
    assert np.all(pooled[0, 1] == 0) and np.all(pooled[1, 0] == 0)
    np.testing.assert_array_equal(pooled[0, 0], tabs[0][5])
    keys, counts = m.unique()
    assert set(keys.tolist()) == {int(m.base[0] + 5), int(m.base[2] + 3), int(m.base[1] + 2), int(m.base[2] + 29)}


def test_bf16_tables_store_bf16_values():
    m = _tiny_static(bf16=True)
    w, _, _, _, _ = m.read_rows(m.global_rows(1, np.arange(70)))
    assert np.all(w.view(np.uint32) & 0xFFFF == 0)


# ------------------------------------------------------------------ interaction

def test_interaction_hand_worked(golden_dir):
    g = _golden(golden_dir, "interaction_tiny.json")
    dense = np.array(g["dense"], np.float32)
    pooled = np.array(g["pooled"], np.float64)
    out, mag = oracle.interact(dense, pooled, T=2, D=2)
    np.testing.assert_array_equal(out, np.array(g["out"]))
    dd, dp, _, _ = oracle.interact_backward(np.array(g["dout"], np.float32), dense, pooled, T=2, D=2)
    np.testing.assert_array_equal(dd, np.array(g["d_dense"]))
    np.testing.assert_array_equal(dp, np.array(g["d_pooled"]))


@pytest.mark.parametrize("T,D", [(4, 16), (26, 128), (1, 4)])
def test_interaction_equals_library_gram(T, D):
    rng = np.random.default_rng(T * 1000 + D)
    B = 5
    dense = rng.standard_normal((B, D)).astype(np.float32)
    pooled = rng.standard_normal((B, T, D))
    out, mag = oracle.interact(dense, pooled, T, D)
    F = T + 1
    ii, jj = np.tril_indices(F, k=-1)  # row-major strict lower triangle: (1,0),(2,0),(2,1),...
    assert out.shape == (B, D + F * (F - 1) // 2)
    for b in range(B):
        X = np.concatenate([dense[b:b + 1].astype(np.float64), pooled[b]], axis=0)
        G = X @ X.T
        np.testing.assert_array_equal(out[b, :D], dense[b].astype(np.float64))
        np.testing.assert_allclose(out[b, D:], G[ii, jj], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(mag[b, D:], (np.abs(X) @ np.abs(X).T)[ii, jj], rtol=1e-12)


def test_interaction_special_cases():
    D, T = 8, 3
    eye = np.eye(D)
    dense = eye[0:1].astype(np.float32)
    pooled = eye[1:4][None]                 # orthonormal vectors: every pair is 0
    out, _ = oracle.interact(dense, pooled, T, D)
    assert np.all(out[0, D:] == 0)
    v = np.arange(1, D + 1, dtype=np.float64)
    pooled = np.stack([v, v, -v])[None]     # x1 = x2 = v, x3 = -v
    out, _ = oracle.interact(np.zeros((1, D), np.float32), pooled, T, D)
    # pairs: (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
    n2 = float(v @ v)
    np.testing.assert_array_equal(out[0, D:], [0, 0, n2, 0, -n2, -n2])


def test_interaction_backward_finite_differences():
    rng = np.random.default_rng(11)
    B, T, D = 2, 3, 4
    F = T + 1
    dense = rng.standard_normal((B, D)).astype(np.float32)
    pooled = rng.standard_normal((B, T, D))
    dout = rng.standard_normal((B, D + F * (F - 1) // 2)).astype(np.float32)
    dd, dp, _, _ = oracle.interact_backward(dout, dense, pooled, T, D)
    ii, jj = np.tril_indices(F, k=-1)

    def loss(X, b):  # sum(dout * out) for one sample, out computed by brute force
        G = X @ X.T
        return float(dout[b, :D].astype(np.float64) @ X[0] + dout[b, D:].astype(np.float64) @ G[ii, jj])

    h = 1e-6
    for b in range(B):
        X = np.concatenate([dense[b:b + 1].astype(np.float64), pooled[b]], axis=0)
        num = np.zeros_like(X)
        for i in range(F):
            for k in range(D):
                Xp, Xm = X.copy(), X.copy()
                Xp[i, k] += h
                Xm[i, k] -= h
                num[i, k] = (loss(Xp, b) - loss(Xm, b)) / (2 * h)
        np.testing.assert_allclose(dd[b], num[0], rtol=1e-7, atol=1e-7)
        np.testing.assert_allclose(dp[b], num[1:], rtol=1e-7, atol=1e-7)


# ------------------------------------------------------------------ Adagrad

def _hashed(dim=1, rowwise=False, lr=0.01, eps=1e-8):
    return oracle.Model(1, dim, hashed=True, capacity=64, rowwise=rowwise, lr=lr, eps=eps,
                        init_acc=0.1, hash_init=0.0, seed=5)


def test_adagrad_single_and_duplicate_steps(golden_dir):
    g = _golden(golden_dir, "adagrad_steps.json")
    for case in g["cases"][:3]:
        m = _hashed(lr=case["lr"], eps=case["eps"])
        n = len(case["grads"])
        ids = np.full(n, 12345, np.int64)       # one key, looked up n times (one bag each)
        pooled, _, flags = m.forward(ids, None, n)
        assert flags == 0 and np.all(pooled == 0)   # new key starts at w = 0
        assert m.backward_adagrad(np.array(case["grads"]).reshape(n, 1, 1)) == 0
        w, acc, _, _, found = m.read_rows([12345])
        assert found[0]
        assert acc[0, 0] == np.float32(Decimal(case["acc1"]))
        ref = float(Decimal(case["w1"]))
        assert abs(float(w[0, 0]) - ref) <= 1.2e-7 * abs(ref)


def test_adagrad_rowwise_step(golden_dir):
    case = _golden(golden_dir, "adagrad_steps.json")["cases"][3]
    m = _hashed(dim=2, rowwise=True, lr=case["lr"])
    m.forward(np.array([7], np.int64), None, 1)
    m.backward_adagrad(np.array(case["grad_row"]).reshape(1, 1, 2))
    w, acc, _, _, _ = m.read_rows([7])
    assert acc.shape == (1, 1) and acc[0, 0] == np.float32(Decimal(case["acc1"]))
    for c in range(2):
        ref = float(Decimal(case["w1"][c]))
        assert abs(float(w[0, c]) - ref) <= 1.2e-7 * abs(ref)


def test_adagrad_mean_pool_scales_gradient():
    # a bag of 4 copies of one key under mean pooling: d(pooled)/d(w) = 4 * 1/4 = 1
    m = oracle.Model(1, 1, hashed=True, capacity=8, mean=True, lr=0.01, seed=1)
    m.forward(np.full(4, 3, np.int64), np.array([0, 4], np.int32), 1)
    m.backward_adagrad(np.ones((1, 1, 1)))
    w, acc, _, _, _ = m.read_rows([3])
    ref = float(Decimal("-0.009534625801546833112161013901347897455324"))
    assert abs(float(w[0, 0]) - ref) <= 1.2e-7 * abs(ref)


def test_untouched_rows_stay_bit_identical_and_touched_rows_change():
    m = _tiny_static()
    before = _dense_tables(m)
    rng = np.random.default_rng(4)
    B = 6
    ids = np.stack([rng.integers(0, m.rows[t], B) for t in range(m.T)], axis=1).reshape(-1)
    m.forward(ids, None, B)
    m.backward_adagrad(rng.standard_normal((B, m.T, m.D)))
    after = _dense_tables(m)
    for t in range(m.T):
        touched = np.zeros(m.rows[t], bool)
        touched[ids[t::m.T]] = True
        assert np.array_equal(after[t][~touched], before[t][~touched])
        assert np.all(np.any(after[t][touched] != before[t][touched], axis=1))


def test_next_forward_sees_updated_rows():
    m = _hashed(dim=3)
    m.forward(np.array([1, 2], np.int64), None, 2)
    m.backward_adagrad(np.array([[[1.0, -2.0, 0.5]], [[0.0, 0.0, 0.0]]]))
    pooled, _, _ = m.forward(np.array([1, 2], np.int64), None, 2)
    w, _, _, _, _ = m.read_rows([1, 2])
    np.testing.assert_array_equal(pooled[:, 0, :], w.astype(np.float64))
    assert np.all(w[1] == 0) and np.all(w[0][[0, 1]] != 0)
    # the signs follow -g
    assert w[0, 0] < 0 < w[0, 1]


def test_backward_without_forward_is_a_state_error():
    m = _hashed()
    assert m.backward_adagrad(np.zeros((1, 1, 1))) == oracle.FLAG_STATE


# ------------------------------------------------------------------ dedup and hash table

def test_unique_matches_numpy():
    w = synth.workload(3, "small")
    m = oracle.Model.from_workload(w)
    b = synth.make_batch(w, 0)
    m.forward(b.ids, b.offsets, b.batch)
    keys, counts = m.unique()
    lens = np.diff(b.offsets)
    table = np.repeat(np.arange(b.batch * w.num_tables) % w.num_tables, lens)
    glob = m.base[table] + b.ids
    uk, uc = np.unique(glob, return_counts=True)
    np.testing.assert_array_equal(keys, uk.astype(np.uint64))
    np.testing.assert_array_equal(counts, uc)


def test_hash_insert_distinct_keys_and_initial_values():
    w = synth.workload(4, "small")
    m = oracle.Model.from_workload(w)
    b = synth.make_batch(w, 0)
    pooled, _, flags = m.forward(b.ids, None, b.batch)
    assert flags == 0
    assert np.all(pooled == 0)                      # every key is new: w = 0
    keys, wv, acc = m.export()
    np.testing.assert_array_equal(keys, np.unique(b.ids).astype(np.uint64))
    assert np.all(wv == 0) and np.all(acc == np.float32(0.1))


def test_hash_negative_key_and_full_table():
    m = oracle.Model(1, 2, hashed=True, capacity=4, seed=1)
    _, _, flags = m.forward(np.array([1, 2, -5], np.int64), None, 3)
    assert flags == oracle.FLAG_BAD_KEY
    assert m.num_rows() == 2
    _, _, flags = m.forward(np.array([3, 4, 5, 1], np.int64), None, 4)
    assert flags == oracle.FLAG_TABLE_FULL
    assert m.num_rows() == 4
    keys, _ = m.unique()
    assert keys.tolist() == [1, 3, 4]


# ------------------------------------------------------------------ admission / eviction

def _one_lookup_step(m, key, g):
    """One backward step in which `key` is looked up once with gradient g (dim 1)."""
    m.forward(np.array([key], np.int64), None, 1)
    assert m.backward_adagrad(np.full((1, 1, 1), g)) == 0


def test_admission_holds_updates_until_the_minimum_count(golden_dir):
    """Reading R19 with minimum 3: the first two steps leave the row at its initial value;
    the third (count 3, this step's lookup included) applies exactly one Adagrad step from the
    initial state, so the row equals the hand-derived single step."""
    single = _golden(golden_dir, "adagrad_steps.json")["cases"][0]
    m = _hashed(lr=single["lr"], eps=single["eps"])
    m.set_admission(3)
    for step in (1, 2):
        _one_lookup_step(m, 7, 1.0)
        w, acc, _, _, found = m.read_rows([7])
        assert found[0] and w[0, 0] == 0.0 and acc[0, 0] == np.float32(0.1)
        freq, last = m.key_stats([7])
        assert freq[0] == step and last[0] == step
    _one_lookup_step(m, 7, 1.0)
    w, acc, _, _, _ = m.read_rows([7])
    assert acc[0, 0] == np.float32(Decimal(single["acc1"]))
    ref = float(Decimal(single["w1"]))
    assert abs(float(w[0, 0]) - ref) <= 1.2e-7 * abs(ref)


def test_admission_counts_every_lookup_of_the_batch(golden_dir):
    """Three lookups of one key in one batch reach a minimum of 3 at once: the summed gradient
    0.5 + 1.5 + 0 gives the hand-derived duplicate step; a key looked up twice stays held."""
    dup = _golden(golden_dir, "adagrad_steps.json")["cases"][1]
    m = _hashed(lr=dup["lr"], eps=dup["eps"])
    m.set_admission(3)
    m.forward(np.array([9, 9, 9, 11, 11], np.int64), None, 5)
    m.backward_adagrad(np.array([0.5, 1.5, 0.0, 2.0, 2.0]).reshape(5, 1, 1))
    w, acc, _, _, _ = m.read_rows([9, 11])
    assert acc[0, 0] == np.float32(Decimal(dup["acc1"]))
    ref = float(Decimal(dup["w1"]))
    assert abs(float(w[0, 0]) - ref) <= 1.2e-7 * abs(ref)
    assert w[1, 0] == 0.0 and acc[1, 0] == np.float32(0.1)
    freq, last = m.key_stats([9, 11, 12])
    assert freq.tolist() == [3, 2, 0] and last.tolist() == [1, 1, 0]


def test_eviction_by_idle_steps_and_by_count():
    """Reading R20: A is looked up in steps 1-3, B in 1-2, C in 1.  After step 3 the idle
    times are 0, 1, 2: max_idle 1 removes C only; C comes back fresh.  A count minimum of 3
    then removes B (2 lookups) but keeps A (3) and the fresh C only if counted 3 times."""
    m = _hashed()
    A, B, C = 101, 202, 303
    for step, keys in enumerate([[A, B, C], [A, B], [A]], start=1):
        m.forward(np.array(keys, np.int64), None, len(keys))
        m.backward_adagrad(np.ones((len(keys), 1, 1)))
    freq, last = m.key_stats([A, B, C])
    assert freq.tolist() == [3, 2, 1] and last.tolist() == [3, 2, 1]
    assert m.evict(0, 0) == 0                     # max_idle 0 and min_count 0: nothing
    assert m.evict(2, 0) == 0                     # idle 2 is not more than 2
    assert m.evict(1, 0) == 1                     # C: idle 2 > 1
    keys, _, _ = m.export()
    assert keys.tolist() == sorted([A, B])
    w, acc, _, _, found = m.read_rows([C])
    assert not found[0]
    pooled, _, _ = m.forward(np.array([C], np.int64), None, 1)
    assert pooled[0, 0, 0] == 0.0                 # a fresh row at the initial value
    m.backward_adagrad(np.ones((1, 1, 1)))
    freq, last = m.key_stats([A, B, C])
    assert freq.tolist() == [3, 2, 1] and last.tolist() == [3, 2, 4]
    assert m.evict(0, 3) == 2                     # B (2) and the fresh C (1)
    keys, _, _ = m.export()
    assert keys.tolist() == [A]


def test_eviction_frees_capacity():
    """Evicted keys no longer count against the table's capacity."""
    m = oracle.Model(1, 1, hashed=True, capacity=2, seed=1)
    m.forward(np.array([1, 2], np.int64), None, 2)
    m.backward_adagrad(np.ones((2, 1, 1)))
    _, _, flags = m.forward(np.array([3], np.int64), None, 1)
    assert flags == oracle.FLAG_TABLE_FULL
    m.backward_adagrad(np.ones((1, 1, 1)))
    assert m.evict(0, 2) == 2                     # both keys were counted once
    _, _, flags = m.forward(np.array([3], np.int64), None, 1)
    assert flags == 0


# ------------------------------------------------------------------ int8 row codec

def test_codec_hand_worked_rounding_to_even():
    """Reading R21 on rows whose scale is exact: max|x| = 127 gives scale 1, max|x| = 63.5
    gives scale 0.5, so every quotient is exact and the codes show the rounding rule (ties to
    even: 62.5 -> 62, -3.5 -> -4, 2.5 -> 2; half away from zero would give 63, -4, 3)."""
    x = np.array([[127.0, 62.5, -3.5, 0.49, -127.0, 2.5],
                  [0.75, 1.25, -63.5, 0.0, 63.5, -0.25]], np.float32)
    q, s = oracle.quantize_rows(x)
    assert s.tolist() == [1.0, 0.5]
    assert q[0].tolist() == [127, 62, -4, 0, -127, 2]
    assert q[1].tolist() == [2, 2, -127, 0, 127, 0]
    d = oracle.dequantize_rows(q, s)
    assert d[0].tolist() == [127.0, 62.0, -4.0, 0.0, -127.0, 2.0]
    assert d[1].tolist() == [1.0, 1.0, -63.5, 0.0, 63.5, 0.0]


def test_codec_zero_row_and_error_bound():
    """A zero row keeps scale 0 and codes 0; on random rows the largest magnitude maps to
    +-127 and every decoded value is within half a step (plus fp32 rounding) of its input."""
    q, s = oracle.quantize_rows(np.zeros((1, 8), np.float32))
    assert s[0] == 0.0 and not q.any()
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((64, 40)) * rng.uniform(0.01, 100, size=(64, 1))).astype(np.float32)
    q, s = oracle.quantize_rows(x)
    amax = np.abs(x).max(axis=1)
    np.testing.assert_allclose(s, amax / 127, rtol=1e-7)
    assert np.all(np.abs(q.astype(np.int64)).max(axis=1) == 127)
    d = oracle.dequantize_rows(q, s)
    assert np.all(np.abs(d - x) <= s[:, None] * 0.5 * (1 + 1e-5) + 1e-30)


# ------------------------------------------------------------------ cross interaction

def test_cross_forward_hand_worked():
    """Reading R22 on exact values: s = xl . w = 0.5 + 0 + 1 = 1.5, out = x0 s + b + xl."""
    x0 = np.array([[1.0, 2.0, 3.0]], np.float32)
    xl = np.array([[0.5, -1.0, 2.0]], np.float32)
    w = np.array([1.0, 0.0, 0.5], np.float32)
    b = np.array([0.25, -0.5, 1.0], np.float32)
    out, mag = oracle.cross_forward(x0, xl, w, b)
    assert out.tolist() == [[2.25, 1.5, 7.5]]
    assert mag.tolist() == [[1.0 * 1.5 + 0.25 + 0.5, 2.0 * 1.5 + 0.5 + 1.0, 3.0 * 1.5 + 1.0 + 2.0]]
    out, _ = oracle.cross_forward(x0, xl, np.zeros(3, np.float32), b)   # w = 0: xl + b
    assert out.tolist() == [(xl[0] + b).tolist()]


def test_cross_backward_exact_directional_derivatives():
    """The layer is linear in each of x0, xl, w, b with the others fixed, so for any
    direction v: L(. + v) - L(.) equals <gradient, v> exactly when every value is a small
    integer (double arithmetic is then exact).  L = sum of dout * out over the batch."""
    rng = np.random.default_rng(22)
    B, K = 5, 7
    ints = lambda *s: rng.integers(-3, 4, size=s).astype(np.float32)
    x0, xl, dout = ints(B, K), ints(B, K), ints(B, K)
    w, b = ints(K), ints(K)
    (dx0, dxl, dw, db), _ = oracle.cross_backward(x0, xl, w, dout)
    L = lambda x0_, xl_, w_, b_: float((oracle.cross_forward(x0_, xl_, w_, b_)[0] * dout).sum())
    base = L(x0, xl, w, b)
    v2, v1 = ints(B, K), ints(K)
    assert L(x0 + v2, xl, w, b) - base == float((dx0 * v2).sum())
    assert L(x0, xl + v2, w, b) - base == float((dxl * v2).sum())
    assert L(x0, xl, w + v1, b) - base == float((dw * v1).sum())
    assert L(x0, xl, w, b + v1) - base == float((db * v1).sum())


# ------------------------------------------------------------------ Adagrad Decay

@pytest.mark.parametrize("rowwise", [False, True])
def test_adagrad_decay_by_period(rowwise):
    """Reading R23 with rate 1/2 and periods of two steps, on exactly representable values
    (initial accumulator 0.5, gradient 1 per element): key 7, updated in steps 1 to 5, has
    accumulators 1.5, 2.5 (period 0: no discount), 2.5/2 + 1 = 2.25, 3.25 (period 1: one
    discount at its start) and 3.25/2 + 1 = 2.625 (period 2); key 9, first updated in step 5,
    starts from 0.5 discounted for periods 1 and 2: 0.5/4 + 1 = 1.125."""
    D = 2 if rowwise else 1
    m = oracle.Model(1, D, hashed=True, capacity=64, rowwise=rowwise, init_acc=0.5, seed=5)
    m.set_adagrad_decay(0.5, 2)
    expect7 = [1.5, 2.5, 2.25, 3.25, 2.625]
    for step in range(5):
        keys = [7] if step < 4 else [7, 9]
        m.forward(np.array(keys, np.int64), None, len(keys))
        m.backward_adagrad(np.ones((len(keys), 1, D)))
        _, acc, _, _, _ = m.read_rows([7])
        assert acc[0, 0] == expect7[step]
    _, acc, _, _, _ = m.read_rows([9])
    assert acc[0, 0] == 1.125
