"""CPU oracle of the sparse embedding layer -- TEST INFRASTRUCTURE ONLY.

A ctypes binding over `oracle.cpp` (plain single-threaded C++, double arithmetic).  Only the
tests, the smoke check and the benchmark's CPU-baseline / reference leg may import this
package.  The CUDA library never links, loads or calls it.

Parity status: every function here is pinned by tests that do not reuse its arithmetic
(brute force in numpy on tiny inputs, closed forms, hand-derived fixtures under
tests/golden/, library special cases, finite differences); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
# a test may point the binding at another build of the same source (planted-mistake runs)
_LIB_OVERRIDE = os.environ.get("ORACLE_LIB")

FLAG_ID_RANGE = 1
FLAG_BAD_KEY = 2
FLAG_TABLE_FULL = 4
FLAG_STATE = 0x100


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ (no FMA contraction, so float steps round one by one)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC",
                               "-ffp-contract=off", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        if _LIB_OVERRIDE:
            L = ctypes.CDLL(_LIB_OVERRIDE)
        else:
            build()
            L = ctypes.CDLL(_LIB)
        p, i64, i32, u64, f32, f64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                      ctypes.c_uint64, ctypes.c_float, ctypes.c_double)
        L.orc_splitmix64.argtypes = [u64, u64]
        L.orc_splitmix64.restype = u64
        L.orc_init_value.argtypes = [u64, i32, i64, i32, f32, f32]
        L.orc_init_value.restype = f32
        L.orc_bf16_rne.argtypes = [f32]
        L.orc_bf16_rne.restype = ctypes.c_uint16
        L.orc_create.argtypes = [i32, p, i32, i32, i64, i32, i32, i32, f64, f64, f32, f32,
                                 f32, f32, u64]
        L.orc_create.restype = p
        L.orc_destroy.argtypes = [p]
        L.orc_num_rows.argtypes = [p]
        L.orc_num_rows.restype = i64
        L.orc_forward.argtypes = [p, p, p, i64, p, p]
        L.orc_forward.restype = ctypes.c_uint32
        L.orc_interact.argtypes = [p, p, p, i64, i32, i32, p, p]
        L.orc_interact_backward.argtypes = [p, p, p, p, i64, i32, i32, p, p, p, p]
        L.orc_backward_adagrad.argtypes = [p, p, p]
        L.orc_backward_adagrad.restype = ctypes.c_uint32
        L.orc_read_rows.argtypes = [p, p, i64, p, p, p, p, p]
        L.orc_unique.argtypes = [p, p, p, i64]
        L.orc_unique.restype = i64
        L.orc_export.argtypes = [p, p, p, p, i64]
        L.orc_export.restype = i64
        L.orc_set_admission.argtypes = [p, ctypes.c_uint32]
        L.orc_set_adagrad_decay.argtypes = [p, f64, i64]
        L.orc_evict.argtypes = [p, ctypes.c_uint32, ctypes.c_uint32]
        L.orc_evict.restype = i64
        L.orc_key_stats.argtypes = [p, p, i64, p, p]
        L.orc_quantize_rows.argtypes = [p, i64, i32, p, p]
        L.orc_cross_forward.argtypes = [p, p, p, p, i64, i32, p, p]
        L.orc_cross_backward.argtypes = [p, p, p, p, i64, i32, p, p, p, p, p, p, p, p]
        L.orc_dequantize_rows.argtypes = [p, p, i64, i32, p]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def splitmix64(seed: int, n: int) -> int:
    return int(lib().orc_splitmix64(seed & (2**64 - 1), n & (2**64 - 1)))


def init_value(seed: int, t: int, row: int, col: int, lo: float = -0.05, hi: float = 0.05) -> np.float32:
    return np.float32(lib().orc_init_value(seed & (2**64 - 1), t, row, col, lo, hi))


def bf16_rne_bits(x: float) -> int:
    return int(lib().orc_bf16_rne(float(np.float32(x))))


def interact(dense: np.ndarray, pooled: np.ndarray, T: int, D: int,
             pooled_mag: Optional[np.ndarray] = None):
    """(out [B, D+P], magnitude [B, D+P]) in float64.  pooled_mag: magnitudes of the pooled
    inputs (from Model.forward); the output magnitude then uses max(|x|, mag) per input."""
    dense = _c(dense, np.float32)
    pooled = _c(pooled, np.float64)
    pm = None if pooled_mag is None else _c(pooled_mag, np.float64)
    B = dense.shape[0]
    F = T + 1
    W = D + F * (F - 1) // 2
    out = np.empty((B, W), np.float64)
    mag = np.empty((B, W), np.float64)
    lib().orc_interact(_ptr(dense), _ptr(pooled), _ptr(pm), B, T, D, _ptr(out), _ptr(mag))
    return out, mag


def interact_backward(dout: np.ndarray, dense: np.ndarray, pooled: np.ndarray, T: int, D: int,
                      pooled_mag: Optional[np.ndarray] = None):
    """(d_dense [B,D], d_pooled [B,T,D], mag_dense, mag_pooled) in float64."""
    dout = _c(dout, np.float32)
    dense = _c(dense, np.float32)
    pooled = _c(pooled, np.float64)
    pm = None if pooled_mag is None else _c(pooled_mag, np.float64)
    B = dense.shape[0]
    dd = np.empty((B, D), np.float64)
    dp = np.empty((B, T, D), np.float64)
    md = np.empty((B, D), np.float64)
    mp = np.empty((B, T, D), np.float64)
    lib().orc_interact_backward(_ptr(dout), _ptr(dense), _ptr(pooled), _ptr(pm), B, T, D,
                                _ptr(dd), _ptr(dp), _ptr(md), _ptr(mp))
    return dd, dp, md, mp


def cross_forward(x0, xl, w, b):
    """One cross layer x0 * (xl . w) + b + xl per sample: (out [B,K], magnitude) float64."""
    x0, xl = _c(x0, np.float32), _c(xl, np.float32)
    w, b = _c(w, np.float32), _c(b, np.float32)
    B, K = x0.shape
    out = np.empty((B, K), np.float64)
    mag = np.empty((B, K), np.float64)
    lib().orc_cross_forward(_ptr(x0), _ptr(xl), _ptr(w), _ptr(b), B, K, _ptr(out), _ptr(mag))
    return out, mag


def cross_backward(x0, xl, w, dout):
    """Gradients of one cross layer: (dx0, dxl [B,K], dw, db [K]) and their magnitudes,
    float64: returns ((dx0, dxl, dw, db), (m_dx0, m_dxl, m_dw, m_db))."""
    x0, xl = _c(x0, np.float32), _c(xl, np.float32)
    w, dout = _c(w, np.float32), _c(dout, np.float32)
    B, K = x0.shape
    g = [np.empty((B, K)), np.empty((B, K)), np.empty(K), np.empty(K)]
    m = [np.empty((B, K)), np.empty((B, K)), np.empty(K), np.empty(K)]
    lib().orc_cross_backward(_ptr(x0), _ptr(xl), _ptr(w), _ptr(dout), B, K,
                             *[_ptr(a) for a in g], *[_ptr(a) for a in m])
    return tuple(g), tuple(m)


def quantize_rows(x: np.ndarray):
    """int8 codes [n, d] and fp32 scales [n] of the rows of x (float32 [n, d])."""
    x = _c(x, np.float32)
    n, d = x.shape
    q = np.empty((n, d), np.int8)
    scale = np.empty(n, np.float32)
    lib().orc_quantize_rows(_ptr(x), n, d, _ptr(q), _ptr(scale))
    return q, scale


def dequantize_rows(q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """float32 rows code * scale."""
    q = _c(q, np.int8)
    scale = _c(scale, np.float32)
    n, d = q.shape
    x = np.empty((n, d), np.float32)
    lib().orc_dequantize_rows(_ptr(q), _ptr(scale), n, d, _ptr(x))
    return x


class Model:
    """Parameter state of one embedding layer (static tables or one hashed table)."""

    def __init__(self, num_tables: int, dim: int, rows=None, hashed: bool = False,
                 capacity: int = 0, bf16: bool = False, mean: bool = False,
                 rowwise: bool = False, lr: float = 0.01, eps: float = 1e-8,
                 init_acc: float = 0.1, lo: float = -0.05, hi: float = 0.05,
                 hash_init: float = 0.0, seed: int = 0):
        self.T, self.D = num_tables, dim
        self.hashed, self.rowwise = hashed, rowwise
        self.rows = None if rows is None else _c(rows, np.int64)
        self.base = None if rows is None else np.concatenate(([0], np.cumsum(self.rows)))
        self._h = lib().orc_create(num_tables, _ptr(self.rows), dim, int(hashed), capacity,
                                   int(bf16), int(mean), int(rowwise), lr, eps, init_acc,
                                   lo, hi, hash_init, seed & (2**64 - 1))

    @classmethod
    def from_workload(cls, w):
        return cls(w.num_tables, w.dim, rows=w.rows, hashed=w.hashed, capacity=w.capacity,
                   bf16=(w.dtype == "bf16"), mean=(w.pooling == "mean"),
                   rowwise=(w.optimizer == "adagrad_row"), lr=w.lr, eps=w.eps,
                   init_acc=w.init_acc, lo=w.init_lo, hi=w.init_hi, hash_init=w.hash_init,
                   seed=w.seed)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().orc_destroy(h)
            self._h = None

    @property
    def acc_width(self) -> int:
        return 1 if self.rowwise else self.D

    def num_rows(self) -> int:
        return int(lib().orc_num_rows(self._h))

    def forward(self, ids: np.ndarray, offsets: Optional[np.ndarray], batch: int):
        """(pooled [B,T,D], magnitude [B,T,D], flags) in float64."""
        ids = _c(ids, np.int64)
        offs = None if offsets is None else _c(offsets, np.int32)
        pooled = np.empty((batch, self.T, self.D), np.float64)
        mag = np.empty((batch, self.T, self.D), np.float64)
        flags = lib().orc_forward(self._h, _ptr(ids), _ptr(offs), batch, _ptr(pooled), _ptr(mag))
        return pooled, mag, int(flags)

    def backward_adagrad(self, d_pooled: np.ndarray, mag: Optional[np.ndarray] = None) -> int:
        d_pooled = _c(d_pooled, np.float64)
        mag = None if mag is None else _c(mag, np.float64)
        return int(lib().orc_backward_adagrad(self._h, _ptr(d_pooled), _ptr(mag)))

    def global_rows(self, table: int, ids) -> np.ndarray:
        return (self.base[table] + np.asarray(ids, np.int64)).astype(np.uint64)

    def read_rows(self, keys):
        """keys: global rows (static) or raw keys (hashed).
        Returns (w [n,D] f32, acc [n,AW] f32, mag_w [n,D], mag_acc [n,AW], found [n] bool);
        mag_w / mag_acc hold, element by element, the magnitude of the update that last wrote
        the element (reading R17; 0 for a row never updated)."""
        keys = _c(np.asarray(keys).astype(np.uint64), np.uint64)
        n = keys.shape[0]
        w = np.empty((n, self.D), np.float32)
        acc = np.empty((n, self.acc_width), np.float32)
        mw = np.empty((n, self.D), np.float64)
        ma = np.empty((n, self.acc_width), np.float64)
        found = np.empty(n, np.int8)
        lib().orc_read_rows(self._h, _ptr(keys), n, _ptr(w), _ptr(acc), _ptr(mw), _ptr(ma),
                            _ptr(found))
        return w, acc, mw, ma, found.astype(bool)

    def unique(self):
        """(keys ascending uint64, counts int64) of the last forward's valid lookups."""
        n = int(lib().orc_unique(self._h, None, None, 0))
        keys = np.empty(n, np.uint64)
        counts = np.empty(n, np.int64)
        lib().orc_unique(self._h, _ptr(keys), _ptr(counts), n)
        return keys, counts

    def set_adagrad_decay(self, rate: float, period_steps: int):
        """Accumulators discounted by `rate` per period of `period_steps` backward steps,
        applied when a row is next updated (0 steps: no decay)."""
        lib().orc_set_adagrad_decay(self._h, float(rate), int(period_steps))

    def set_admission(self, min_count: int):
        """Hashed tables: a key's row is updated only once it has been looked up at least
        min_count times over all steps (0 or 1: at once)."""
        lib().orc_set_admission(self._h, int(min_count))

    def evict(self, max_idle: int, min_count: int) -> int:
        """Hashed tables: remove keys idle for more than max_idle backward steps
        (max_idle > 0) or looked up fewer than min_count times; returns how many."""
        return int(lib().orc_evict(self._h, int(max_idle), int(min_count)))

    def key_stats(self, keys):
        """(lookup counts uint64, last counting step int64) of hashed keys (0, 0: absent)."""
        keys = _c(np.asarray(keys).astype(np.uint64), np.uint64)
        n = keys.shape[0]
        freq = np.empty(n, np.uint64)
        last = np.empty(n, np.int64)
        lib().orc_key_stats(self._h, _ptr(keys), n, _ptr(freq), _ptr(last))
        return freq, last

    def export(self):
        """(keys ascending, w, acc) of every materialised row."""
        n = int(lib().orc_export(self._h, None, None, None, 0))
        keys = np.empty(n, np.uint64)
        w = np.empty((n, self.D), np.float32)
        acc = np.empty((n, self.acc_width), np.float32)
        lib().orc_export(self._h, _ptr(keys), _ptr(w), _ptr(acc), n)
        return keys, w, acc
