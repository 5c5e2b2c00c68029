"""Seeded synthetic inputs for the sparse-embedding hot path.

This module only draws inputs: feature IDs, bag lengths, dense vectors and upstream
gradients.  It holds none of the embedding arithmetic (no lookup, pooling, interaction
or optimiser step), so both the CPU oracle and the CUDA path can be fed from it without
sharing any method code.

The five workloads stand in for the DLRM / Criteo-shaped workloads the pages describe
(Merlin Distributed Embeddings article, "Criteo DLRM benchmark" and "synthetic model
benchmark" sections: global batch 65536, Adagrad; HugeCTR interview, section 2: 26-ish
categorical fields mapped through embedding tables).  The Criteo click logs themselves are
not available, so the distributions below (Zipf over a seeded permutation of ranks,
Poisson bag lengths, N(0,1) dense inputs and gradients) replace them.

Random streams: every purpose (ids, lengths, dense, dout, permutation, keys) draws from
its own numpy PCG64 stream seeded with (config seed, purpose tag, step, table).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# purpose tags of the independent random streams
TAG_IDS, TAG_LEN, TAG_DENSE, TAG_DOUT, TAG_PERM, TAG_KEYS = 1, 2, 3, 4, 5, 6

MASK63 = (1 << 63) - 1


def config_seed(k: int) -> int:
    """Seed of workload k (1-based): 0x5EED0000 + k."""
    return 0x5EED0000 + k


def _rng(seed: int, *words: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *words])))


@dataclasses.dataclass
class Workload:
    """Shape and distribution of one synthetic workload.

    ids_dist: "uniform" (i.i.d. over the table), "zipf" (rank ~ Zipf(alpha) over the
    table, mapped through a seeded permutation), or "zipf_keys" (hashed config: rank ~
    Zipf(alpha) over `num_keys` distinct keys, mapped by a 63-bit bijection to int64 keys).
    bag: "one" (one ID per (sample, table)), "uniform_1_4", or "poisson" (1+Poisson(mu)
    capped at `bag_cap`).
    """

    name: str
    batch: int
    num_tables: int
    dim: int
    rows: Optional[list]            # rows per table (static tables) or None (hashed)
    dtype: str = "f32"              # "f32" | "bf16"
    pooling: str = "sum"            # "sum" | "mean"
    optimizer: str = "adagrad"      # "adagrad" (per element) | "adagrad_row"
    lr: float = 0.01
    eps: float = 1e-8
    init_acc: float = 0.1
    interaction: bool = False
    ids_dist: str = "uniform"
    alpha: float = 1.0
    bag: str = "one"
    bag_mu: float = 19.0
    bag_cap: int = 100
    hashed: bool = False
    capacity: int = 0
    num_keys: int = 0
    steps: int = 1
    seed: int = 0
    init_lo: float = -0.05
    init_hi: float = 0.05
    hash_init: float = 0.0

    @property
    def num_features(self) -> int:
        """F = T + 1 interaction vectors (dense first)."""
        return self.num_tables + 1

    @property
    def num_pairs(self) -> int:
        f = self.num_features
        return f * (f - 1) // 2

    @property
    def out_width(self) -> int:
        return self.dim + self.num_pairs

    @property
    def multi_hot(self) -> bool:
        return self.bag != "one"

    def max_lookups(self) -> int:
        if self.bag == "one":
            return self.batch * self.num_tables
        if self.bag == "uniform_1_4":
            return self.batch * self.num_tables * 4
        return self.batch * self.num_tables * self.bag_cap


def criteo_rows() -> list:
    """Row counts of the Criteo-shaped workload: 8 tables of 10M rows, then 18 tables
    log-spaced from 100 to 1M rows (round(100 * 10**(4k/17)), k = 0..17)."""
    return [10_000_000] * 8 + [int(round(100 * 10 ** (4 * k / 17))) for k in range(18)]


def workload(k: int, scale: str = "full") -> Workload:
    """The five workloads; scale="small" gives a shrunken copy (same generators, fewer
    rows and samples, batch chosen to leave ragged tails) that the oracle finishes in
    seconds."""
    small = scale == "small"
    s = config_seed(k)
    if k == 1:
        return Workload("tiny-dlrm-4x1000x16-b64", batch=64, num_tables=4, dim=16,
                        rows=[1000] * 4, interaction=True, ids_dist="uniform",
                        bag="uniform_1_4", seed=s)
    if k == 2:
        rows = criteo_rows()
        batch = 65536
        if small:
            rows = [max(100, r // 1000) for r in rows]
            batch = 1000
        return Workload("criteo-onehot-26x128-b65536" if not small else "criteo-onehot-small",
                        batch=batch, num_tables=26, dim=128, rows=rows, interaction=True,
                        ids_dist="zipf", alpha=1.05, bag="one", seed=s)
    if k == 3:
        rows = [2_000_000] * 26
        batch = 16384
        if small:
            rows = [20_000] * 26
            batch = 333
        return Workload("multihot-bf16-26x2Mx64-b16384" if not small else "multihot-bf16-small",
                        batch=batch, num_tables=26, dim=64, rows=rows, dtype="bf16",
                        pooling="mean", optimizer="adagrad_row", lr=0.02,
                        ids_dist="zipf", alpha=1.1, bag="poisson", bag_mu=19.0,
                        bag_cap=100, seed=s)
    if k == 4:
        if small:
            return Workload("hashed-ev-small", batch=300, num_tables=40, dim=32, rows=None,
                            hashed=True, capacity=1 << 15, num_keys=20_000,
                            ids_dist="zipf_keys", alpha=1.1, steps=4, seed=s)
        return Workload("hashed-ev-64Mslots-d32-b32768x40", batch=32768, num_tables=40,
                        dim=32, rows=None, hashed=True, capacity=1 << 26,
                        num_keys=50_000_000, ids_dist="zipf_keys", alpha=1.1, steps=20,
                        seed=s)
    if k == 5:
        rows = [4_000_000] * 26
        batch = 262144
        if small:
            rows = [40_000] * 26
            batch = 1531
        return Workload("bandwidth-stress-26x4Mx128-b262144" if not small else "bandwidth-stress-small",
                        batch=batch, num_tables=26, dim=128, rows=rows, interaction=True,
                        ids_dist="uniform", bag="one", steps=10, seed=s)
    raise ValueError(f"no workload {k}")


# ---------------------------------------------------------------------------------------
# samplers

def zipf_ranks(rng: np.random.Generator, n_items: int, alpha: float, size: int) -> np.ndarray:
    """Ranks k in [1, n_items] with P(k) proportional to k**-alpha.

    Rejection-inversion (Hormann & Derflinger, "Rejection-inversion to generate variates
    from monotone discrete distributions", ACM TOMACS 6(3), 1996), vectorised: invert the
    integral H of the hat x**-alpha over [1.5 - 1, n + 0.5], round to the nearest integer
    and accept by the squeeze test or the exact test against H(k + 0.5) - k**-alpha.
    """
    if n_items < 1:
        raise ValueError("n_items must be >= 1")
    if n_items == 1:
        return np.ones(size, dtype=np.int64)
    a = float(alpha)
    om = 1.0 - a

    def helper1(x):  # log1p(x) / x, continuous at 0
        out = np.ones_like(x)
        nz = np.abs(x) > 1e-8
        out[nz] = np.log1p(x[nz]) / x[nz]
        out[~nz] = 1.0 - x[~nz] * (0.5 - x[~nz] * (1.0 / 3.0))
        return out

    def helper2(x):  # expm1(x) / x, continuous at 0
        out = np.ones_like(x)
        nz = np.abs(x) > 1e-8
        out[nz] = np.expm1(x[nz]) / x[nz]
        out[~nz] = 1.0 + x[~nz] * 0.5 * (1.0 + x[~nz] * (1.0 / 3.0))
        return out

    def H(x):
        lx = np.log(x)
        return helper2(om * lx) * lx

    def H_inv(y):
        t = np.maximum(y * om, -1.0)
        return np.exp(helper1(t) * y)

    def h(x):
        return np.exp(-a * np.log(x))

    hx1 = H(np.array([1.5]))[0] - 1.0
    hn = H(np.array([n_items + 0.5]))[0]
    s = 2.0 - H_inv(np.array([H(np.array([2.5]))[0] - h(np.array([2.0]))[0]]))[0]

    out = np.empty(size, dtype=np.int64)
    todo = np.arange(size)
    while todo.size:
        u = hn + rng.random(todo.size) * (hx1 - hn)
        x = H_inv(u)
        k = np.clip(np.floor(x + 0.5), 1, n_items)
        ok = (k - x <= s) | (u >= H(k + 0.5) - h(k))
        out[todo[ok]] = k[ok].astype(np.int64)
        todo = todo[~ok]
    return out


def key_bijection(rank: np.ndarray, seed: int) -> np.ndarray:
    """A seeded bijection of [0, 2**63) (odd multipliers and xor-shifts, all taken mod
    2**63), used to turn Zipf ranks of the hashed workload into raw int64 keys.  The
    all-ones 64-bit pattern (-1) can never come out, since every result is < 2**63."""
    m = np.uint64(MASK63)
    x = (rank.astype(np.uint64) + np.uint64((seed * 0x9E3779B97F4A7C15) & MASK63)) & m
    x = (x * np.uint64(0xD6E8FEB86659FD93 | 1)) & m
    x ^= x >> np.uint64(31)
    x = (x * np.uint64(0xA0761D6478BD642F | 1)) & m
    x ^= x >> np.uint64(29)
    return x.astype(np.int64)


# ---------------------------------------------------------------------------------------
# batches

@dataclasses.dataclass
class Batch:
    ids: np.ndarray                 # int64 [nnz], bag-major (bag = b*T + t), table-local IDs or keys
    offsets: Optional[np.ndarray]   # int32 [B*T+1] for multi-hot, None for one-hot
    dense: Optional[np.ndarray]     # float32 [B, D] (interaction workloads)
    dout: np.ndarray                # float32 [B, D+P] (interaction) or [B, T, D] (pooled grad)
    batch: int

    @property
    def nnz(self) -> int:
        return int(self.ids.shape[0])


_perm_cache: dict = {}


def _rank_to_id(w: Workload, t: int, ranks0: np.ndarray) -> np.ndarray:
    """Zero-based ranks -> table-local IDs through a seeded permutation of [0, rows)."""
    n = w.rows[t]
    key = (w.seed, t, n)
    perm = _perm_cache.get(key)
    if perm is None:
        perm = _rng(w.seed, TAG_PERM, t).permutation(n).astype(np.int64)
        if len(_perm_cache) > 64:
            _perm_cache.clear()
        _perm_cache[key] = perm
    return perm[ranks0]


def _draw_ids(w: Workload, t: int, step: int, count: int) -> np.ndarray:
    rng = _rng(w.seed, TAG_IDS, step, t)
    if w.ids_dist == "uniform":
        return rng.integers(0, w.rows[t], size=count, dtype=np.int64)
    if w.ids_dist == "zipf":
        return _rank_to_id(w, t, zipf_ranks(rng, w.rows[t], w.alpha, count) - 1)
    raise ValueError(w.ids_dist)


def bag_lengths(w: Workload, step: int) -> np.ndarray:
    """Bag length per (sample, table), bag-major [B*T]."""
    n_bags = w.batch * w.num_tables
    if w.bag == "one":
        return np.ones(n_bags, dtype=np.int64)
    rng = _rng(w.seed, TAG_LEN, step)
    if w.bag == "uniform_1_4":
        return rng.integers(1, 5, size=n_bags, dtype=np.int64)
    if w.bag == "poisson":
        return np.minimum(1 + rng.poisson(w.bag_mu, size=n_bags), w.bag_cap).astype(np.int64)
    raise ValueError(w.bag)


def make_batch(w: Workload, step: int = 0, batch: Optional[int] = None) -> Batch:
    """Inputs of one step.  `batch` overrides the workload's batch size (same streams, so
    a smaller batch is not a prefix of the larger one)."""
    if batch is not None:
        w = dataclasses.replace(w, batch=batch)
    B, T, D = w.batch, w.num_tables, w.dim
    if w.hashed:
        rng = _rng(w.seed, TAG_KEYS, step)
        ranks0 = zipf_ranks(rng, w.num_keys, w.alpha, B * T) - 1
        ids = key_bijection(ranks0, w.seed)
        offsets = None
    else:
        lens = bag_lengths(w, step)
        lens_bt = lens.reshape(B, T)
        ids = np.empty(int(lens.sum()), dtype=np.int64)
        offs = np.zeros(B * T + 1, dtype=np.int64)
        np.cumsum(lens, out=offs[1:])
        for t in range(T):
            cnt = int(lens_bt[:, t].sum())
            draws = _draw_ids(w, t, step, cnt)
            if w.bag == "one":
                ids[t::T] = draws
            else:
                # positions of table t's lookups, bag by bag in sample order
                starts = offs[:-1].reshape(B, T)[:, t]
                ln = lens_bt[:, t]
                pos = np.repeat(starts - np.concatenate(([0], np.cumsum(ln)[:-1])), ln) + np.arange(cnt)
                ids[pos] = draws
        offsets = None if w.bag == "one" else offs.astype(np.int32)
    dense = None
    if w.interaction:
        dense = _rng(w.seed, TAG_DENSE, step).standard_normal((B, D), dtype=np.float32)
        dout = _rng(w.seed, TAG_DOUT, step).standard_normal((B, w.out_width), dtype=np.float32)
    else:
        dout = _rng(w.seed, TAG_DOUT, step).standard_normal((B, T, D), dtype=np.float32)
    return Batch(ids=ids, offsets=offsets, dense=dense, dout=dout, batch=B)


def zipf_expected_unique(n_items: int, alpha: float, draws: int) -> float:
    """Expected number of distinct ranks among `draws` Zipf draws: sum_k 1-(1-p_k)^n."""
    k = np.arange(1, n_items + 1, dtype=np.float64)
    p = k ** -alpha
    p /= p.sum()
    return float(np.sum(-np.expm1(draws * np.log1p(-p))))
