"""GB300-native sparse embedding layer for DLRM-style recommenders.

A thin ctypes binding over libemb.so, the CUDA library declared in include/emb.h.  Every
method marshals its arguments (torch tensors -> device pointers, the current CUDA stream)
and calls the C entry point of the same name; all arithmetic runs in the library's
kernels.  There is no CPU path: if libemb.so is missing this package fails to import.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libemb.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()' or "
        "python recommender_model_embedding_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)

EMB_OK, EMB_EINVAL, EMB_ENOMEM, EMB_ESTATE, EMB_ECUDA = 0, 1, 2, 3, 4
FLAG_ID_RANGE, FLAG_BAD_KEY, FLAG_TABLE_FULL, FLAG_BAD_OFFSETS = 0x1, 0x2, 0x4, 0x8
FLAG_WAIT_LIMIT = 0x10
F32, BF16 = 0, 1
POOL_SUM, POOL_MEAN = 0, 1
ADAGRAD, ADAGRAD_ROWWISE = 0, 1


class EmbConfig(ctypes.Structure):
    _fields_ = [("num_tables", ctypes.c_int32), ("dim", ctypes.c_int32),
                ("rows", ctypes.POINTER(ctypes.c_int64)), ("hashed", ctypes.c_int32),
                ("capacity", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("pooling", ctypes.c_int32), ("optimizer", ctypes.c_int32),
                ("lr", ctypes.c_float), ("eps", ctypes.c_float), ("init_acc", ctypes.c_float),
                ("init_lo", ctypes.c_float), ("init_hi", ctypes.c_float),
                ("hash_init", ctypes.c_float), ("seed", ctypes.c_uint64),
                ("max_batch", ctypes.c_int64), ("max_lookups", ctypes.c_int64)]


_P, _I64, _I32, _U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
_SIGS = {
    "emb_status_str": ([ctypes.c_int], ctypes.c_char_p),
    "emb_create": ([ctypes.POINTER(EmbConfig), ctypes.POINTER(_P)], ctypes.c_int),
    "emb_create_tiered": ([ctypes.POINTER(EmbConfig), _I64, ctypes.POINTER(_P)], ctypes.c_int),
    "emb_destroy": ([_P], None),
    "emb_forward": ([_P, _P, _P, _I64, _I64, _P, _P], ctypes.c_int),
    "emb_interact": ([_P, _P, _P, _I64, _P, _P], ctypes.c_int),
    "emb_interact_backward": ([_P, _P, _P, _P, _I64, _P, _P, _P], ctypes.c_int),
    "emb_backward_adagrad": ([_P, _P, _P], ctypes.c_int),
    "emb_forward_interact": ([_P, _P, _P, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "emb_backward_interact_adagrad": ([_P, _P, _P, _P, _P], ctypes.c_int),
    "emb_train_step_host": ([_P, _P, _P, _I64, _I64, _P, _P, _P, _P, _P], ctypes.c_int),
    "emb_get_status": ([_P, _P, ctypes.POINTER(_U32)], ctypes.c_int),
    "emb_read_rows": ([_P, _I32, _P, _I64, _P, _P, _P], ctypes.c_int),
    "emb_read_unique": ([_P, _P, _P, _I64, ctypes.POINTER(_I64)], ctypes.c_int),
    "emb_export_hash": ([_P, _P, _P, _P, _I64, ctypes.POINTER(_I64)], ctypes.c_int),
    "emb_profile": ([_P, _I32], ctypes.c_int),
    "emb_profile_read": ([_P, _I32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                          ctypes.POINTER(_I64)], ctypes.c_int),
    "emb_profile_reset": ([_P], ctypes.c_int),
    "emb_launch_count": ([_P], _I64),
    "emb_step_tracks_once": ([_P], _I32),
    "emb_set_admission": ([_P, _U32], ctypes.c_int),
    "emb_set_adagrad_decay": ([_P, ctypes.c_float, _U32], ctypes.c_int),
    "emb_quantize_rows": ([_P, _I64, _I32, _P, _P, _P], ctypes.c_int),
    "emb_cross_forward": ([_P, _P, _P, _P, _I64, _I32, _P, _P], ctypes.c_int),
    "emb_cross_backward": ([_P, _P, _P, _P, _I64, _I32, _P, _P, _P, _P, _P], ctypes.c_int),
    "emb_dequantize_rows": ([_P, _P, _I64, _I32, _P, _P], ctypes.c_int),
    "emb_evict": ([_P, _U32, _U32, _P, ctypes.POINTER(_I64)], ctypes.c_int),
    "emb_read_key_stats": ([_P, _P, _I64, _P, _P], ctypes.c_int),
    "emb_prefetch": ([_P, _P, _P, _I64, _I64, _P], ctypes.c_int),
    "emb_set_tier_watermark": ([_P, _I64, _I64], ctypes.c_int),
    "emb_tier_occupancy": ([_P, ctypes.POINTER(_I64)], ctypes.c_int),
    "emb_unique_keys_noalloc": ([_P, _I64, _P, _P, _P, _P], ctypes.c_int),
}
NOALLOC_MAX_KEYS = 524288


CROSS_MAX_K = 9216


def cross_forward(x0, xl, w, b, out, stream=None):
    """One cross layer: out = x0 * (xl . w) + b + xl per sample (CUDA tensors [B, K], [K])."""
    B, K = x0.shape
    _check("emb_cross_forward",
           _lib.emb_cross_forward(_dptr(x0, "f32", B * K, "x0"), _dptr(xl, "f32", B * K, "xl"),
                                  _dptr(w, "f32", K, "w"), _dptr(b, "f32", K, "b"), B, K,
                                  _dptr(out, "f32", B * K, "out"), _stream(stream)))


def cross_backward(x0, xl, w, dout, dx0, dxl, dw, db, stream=None):
    """Gradients of one cross layer (dw, db overwritten); CUDA tensors, asynchronous."""
    B, K = x0.shape
    _check("emb_cross_backward",
           _lib.emb_cross_backward(_dptr(x0, "f32", B * K, "x0"), _dptr(xl, "f32", B * K, "xl"),
                                   _dptr(w, "f32", K, "w"), _dptr(dout, "f32", B * K, "dout"), B, K,
                                   _dptr(dx0, "f32", B * K, "dx0"), _dptr(dxl, "f32", B * K, "dxl"),
                                   _dptr(dw, "f32", K, "dw"), _dptr(db, "f32", K, "db"),
                                   _stream(stream)))


def quantize_rows(x, q, scale, stream=None):
    """int8 codes `q` (int8 [n, d]) and per-row scales `scale` (float32 [n]) of the rows of
    `x` (float32 [n, d]); CUDA tensors, asynchronous."""
    n, d = x.shape
    _check("emb_quantize_rows",
           _lib.emb_quantize_rows(_dptr(x, "f32", n * d, "x"), n, d, _dptr(q, "i8", n * d, "q"),
                                  _dptr(scale, "f32", n, "scale"), _stream(stream)))


def dequantize_rows(q, scale, x, stream=None):
    """x = code * scale row by row (CUDA tensors, asynchronous)."""
    n, d = q.shape
    _check("emb_dequantize_rows",
           _lib.emb_dequantize_rows(_dptr(q, "i8", n * d, "q"), _dptr(scale, "f32", n, "scale"),
                                    n, d, _dptr(x, "f32", n * d, "x"), _stream(stream)))


def unique_keys_noalloc(keys, unique, inverse, num_unique, stream=None):
    """Unique keys of `keys` (int64 CUDA tensor) into `unique` (int64, same length),
    `inverse` (int32, same length) and `num_unique` (int32, one element), with no device
    allocation (scratch lives in the library's fixed device array).  Asynchronous."""
    n = keys.numel()
    _check("emb_unique_keys_noalloc",
           _lib.emb_unique_keys_noalloc(_dptr(keys, "i64", n, "keys"), n,
                                        _dptr(unique, "i64", n, "unique"),
                                        _dptr(inverse, "i32", n, "inverse"),
                                        _dptr(num_unique, "i32", 1, "num_unique"), _stream(stream)))
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res


class EmbError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} failed: {status_str(status)} ({status})")
        self.status = status


def status_str(s: int) -> str:
    return _lib.emb_status_str(int(s)).decode()


def _check(call: str, st: int):
    if st != EMB_OK:
        raise EmbError(call, st)


_DTYPES = {"i64": "int64", "i32": "int32", "f32": "float32", "i8": "int8"}


def _dptr(t, dtype: Optional[str] = None, numel: int = 0, name: str = "tensor") -> Optional[int]:
    """Device pointer of a contiguous CUDA tensor (None passes NULL).  With dtype ("i64",
    "i32", "f32", "i8") and numel, the tensor must have that element type and at least that
    many elements; a mismatch raises ValueError before anything reaches the device (a short
    or mistyped buffer would otherwise be read or written past its end)."""
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA tensor")
    if dtype is not None and str(t.dtype) != "torch." + _DTYPES[dtype]:
        raise ValueError(f"{name}: expected dtype {_DTYPES[dtype]}, got {t.dtype}")
    if t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, at least {numel} needed")
    return t.data_ptr()


def _hptr(a, dtype: Optional[str] = None, numel: int = 0, name: str = "array") -> Optional[int]:
    """Host pointer of a contiguous numpy array or CPU tensor (None passes NULL), with the
    same dtype and size checks as _dptr."""
    if a is None:
        return None
    if hasattr(a, "ctypes"):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError(f"{name}: expected a C-contiguous array")
        if dtype is not None and str(a.dtype) != _DTYPES[dtype]:
            raise ValueError(f"{name}: expected dtype {_DTYPES[dtype]}, got {a.dtype}")
        if a.size < numel:
            raise ValueError(f"{name}: {a.size} elements, at least {numel} needed")
        return a.ctypes.data
    if a.is_cuda or not a.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CPU tensor")
    if dtype is not None and str(a.dtype) != "torch." + _DTYPES[dtype]:
        raise ValueError(f"{name}: expected dtype {_DTYPES[dtype]}, got {a.dtype}")
    if a.numel() < numel:
        raise ValueError(f"{name}: {a.numel()} elements, at least {numel} needed")
    return a.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class EmbCtx:
    """One embedding layer (tables, accumulators, workspace) owned by libemb.so."""

    def __init__(self, num_tables: int, dim: int, rows: Optional[Sequence[int]] = None,
                 hashed: bool = False, capacity: int = 0, dtype: int = F32,
                 pooling: int = POOL_SUM, optimizer: int = ADAGRAD, lr: float = 0.01,
                 eps: float = 1e-8, init_acc: float = 0.1, init_lo: float = -0.05,
                 init_hi: float = 0.05, hash_init: float = 0.0, seed: int = 0,
                 max_batch: int = 1, max_lookups: int = 1, cache_rows: int = 0):
        self._h = None
        self.T, self.D = num_tables, dim
        self.hashed = bool(hashed)
        self.rowwise = optimizer == ADAGRAD_ROWWISE
        rows_arr = None
        if rows is not None:
            rows_arr = (ctypes.c_int64 * len(rows))(*[int(r) for r in rows])
        cfg = EmbConfig(num_tables, dim,
                        ctypes.cast(rows_arr, ctypes.POINTER(ctypes.c_int64)) if rows_arr else None,
                        int(hashed), int(capacity), int(dtype), int(pooling), int(optimizer),
                        lr, eps, init_acc, init_lo, init_hi, hash_init,
                        int(seed) & (2**64 - 1), int(max_batch), int(max_lookups))
        h = _P()
        if cache_rows > 0:  # tiered static tables: host tier plus an HBM cache of cache_rows
            _check("emb_create_tiered", _lib.emb_create_tiered(ctypes.byref(cfg), int(cache_rows),
                                                               ctypes.byref(h)))
        else:
            _check("emb_create", _lib.emb_create(ctypes.byref(cfg), ctypes.byref(h)))
        self._h = h
        self.F = num_tables + 1
        self.out_width = dim + self.F * (self.F - 1) // 2
        self._last = ("", 0)  # kind and batch of the last forward (sizes of its backward)

    @classmethod
    def from_workload(cls, w, max_batch: Optional[int] = None, max_lookups: Optional[int] = None,
                      cache_rows: int = 0):
        """Context for a workload description (any object with the fields of synth.Workload);
        cache_rows > 0: static tables in the host tier with an HBM cache of that many rows."""
        return cls(w.num_tables, w.dim, rows=w.rows, hashed=w.hashed, capacity=w.capacity,
                   dtype=BF16 if w.dtype == "bf16" else F32,
                   pooling=POOL_MEAN if w.pooling == "mean" else POOL_SUM,
                   optimizer=ADAGRAD_ROWWISE if w.optimizer == "adagrad_row" else ADAGRAD,
                   lr=w.lr, eps=w.eps, init_acc=w.init_acc, init_lo=w.init_lo,
                   init_hi=w.init_hi, hash_init=w.hash_init, seed=w.seed,
                   max_batch=max_batch or w.batch, max_lookups=max_lookups or w.max_lookups(),
                   cache_rows=cache_rows)

    def close(self):
        if self._h:
            _lib.emb_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # ---- compute calls (stream-ordered, asynchronous) ----
    # Every tensor is checked for dtype and size against the call's layout before the
    # library sees its pointer (the library trusts the caller's buffers).
    def _lookups(self, ids, offsets, batch: int):
        nnz = ids.numel()
        if offsets is not None:
            _dptr(offsets, "i32", batch * self.T + 1, "offsets")
        elif nnz != batch * self.T:
            raise ValueError(f"ids: {nnz} elements for a one-hot batch of {batch} x {self.T}")
        _dptr(ids, "i64", nnz, "ids")
        return nnz

    def forward(self, ids, offsets, batch: int, pooled, stream=None):
        nnz = self._lookups(ids, offsets, batch)
        _check("emb_forward", _lib.emb_forward(self._h, _dptr(ids), _dptr(offsets), nnz, batch,
                                               _dptr(pooled, "f32", batch * self.T * self.D, "pooled"),
                                               _stream(stream)))
        self._last = ("forward", batch)

    def interact(self, dense, pooled, batch: int, out, stream=None):
        _check("emb_interact",
               _lib.emb_interact(self._h, _dptr(dense, "f32", batch * self.D, "dense"),
                                 _dptr(pooled, "f32", batch * self.T * self.D, "pooled"), batch,
                                 _dptr(out, "f32", batch * self.out_width, "out"), _stream(stream)))

    def interact_backward(self, dout, dense, pooled, batch: int, ddense, dpooled, stream=None):
        BD, BTD = batch * self.D, batch * self.T * self.D
        _check("emb_interact_backward",
               _lib.emb_interact_backward(self._h, _dptr(dout, "f32", batch * self.out_width, "dout"),
                                          _dptr(dense, "f32", BD, "dense"),
                                          _dptr(pooled, "f32", BTD, "pooled"), batch,
                                          _dptr(ddense, "f32", BD, "ddense"),
                                          _dptr(dpooled, "f32", BTD, "dpooled"), _stream(stream)))

    def backward_adagrad(self, dpooled, stream=None):
        kind, batch = self._last
        need = batch * self.T * self.D if kind == "forward" else 0
        _check("emb_backward_adagrad",
               _lib.emb_backward_adagrad(self._h, _dptr(dpooled, "f32", need, "dpooled"),
                                         _stream(stream)))

    def forward_interact(self, ids, offsets, batch: int, dense, out, stream=None):
        nnz = self._lookups(ids, offsets, batch)
        _check("emb_forward_interact",
               _lib.emb_forward_interact(self._h, _dptr(ids), _dptr(offsets), nnz, batch,
                                         _dptr(dense, "f32", batch * self.D, "dense"),
                                         _dptr(out, "f32", batch * self.out_width, "out"),
                                         _stream(stream)))
        self._last = ("forward_interact", batch)

    def backward_interact_adagrad(self, dout, dense, ddense, stream=None):
        kind, batch = self._last
        b = batch if kind == "forward_interact" else 0
        _check("emb_backward_interact_adagrad",
               _lib.emb_backward_interact_adagrad(self._h, _dptr(dout, "f32", b * self.out_width, "dout"),
                                                  _dptr(dense, "f32", b * self.D, "dense"),
                                                  _dptr(ddense, "f32", b * self.D, "ddense"),
                                                  _stream(stream)))

    def train_step_host(self, ids, offsets, batch: int, dense, dout, out, ddense, stream=None):
        """Host buffers (pinned CPU tensors or numpy arrays); asynchronous on `stream`."""
        nnz = int(ids.shape[0])
        if offsets is None and nnz != batch * self.T:
            raise ValueError(f"ids: {nnz} elements for a one-hot batch of {batch} x {self.T}")
        W = self.out_width
        _check("emb_train_step_host",
               _lib.emb_train_step_host(self._h, _hptr(ids, "i64", nnz, "ids"),
                                        _hptr(offsets, "i32", batch * self.T + 1, "offsets"), nnz,
                                        batch, _hptr(dense, "f32", batch * self.D, "dense"),
                                        _hptr(dout, "f32", batch * W, "dout"),
                                        _hptr(out, "f32", batch * W, "out"),
                                        _hptr(ddense, "f32", batch * self.D, "ddense"),
                                        _stream(stream)))

    # ---- synchronous queries ----
    def get_status(self, stream=None) -> int:
        f = _U32(0)
        _check("emb_get_status", _lib.emb_get_status(self._h, _stream(stream), ctypes.byref(f)))
        return int(f.value)

    def read_rows(self, table: int, ids):
        """(w [n, D] float32, acc [n, D or 1] float32, found [n] bool) as numpy arrays."""
        import numpy as np
        ids = np.ascontiguousarray(ids, dtype=np.int64)
        n = ids.shape[0]
        w = np.empty((n, self.D), np.float32)
        acc = np.empty((n, 1 if self.rowwise else self.D), np.float32)
        found = np.empty(n, np.int8)
        _check("emb_read_rows", _lib.emb_read_rows(self._h, table, _hptr(ids), n, _hptr(w),
                                                   _hptr(acc), _hptr(found)))
        return w, acc, found.astype(bool)

    def read_unique(self):
        """(keys int64 [U], counts int32 [U]) of the last forward, in no fixed order."""
        import numpy as np
        U = _I64(0)
        _check("emb_read_unique", _lib.emb_read_unique(self._h, None, None, 0, ctypes.byref(U)))
        keys = np.empty(U.value, np.int64)
        counts = np.empty(U.value, np.int32)
        _check("emb_read_unique", _lib.emb_read_unique(self._h, _hptr(keys), _hptr(counts),
                                                       U.value, ctypes.byref(U)))
        return keys, counts

    def export_hash(self):
        """(keys int64 [n], w [n, D], acc [n, D or 1]) of every occupied slot."""
        import numpy as np
        n = _I64(0)
        _check("emb_export_hash", _lib.emb_export_hash(self._h, None, None, None, 0, ctypes.byref(n)))
        cap = n.value
        keys = np.empty(cap, np.int64)
        w = np.empty((cap, self.D), np.float32)
        acc = np.empty((cap, 1 if self.rowwise else self.D), np.float32)
        _check("emb_export_hash", _lib.emb_export_hash(self._h, _hptr(keys), _hptr(w), _hptr(acc),
                                                       cap, ctypes.byref(n)))
        return keys[:min(cap, n.value)], w[:min(cap, n.value)], acc[:min(cap, n.value)]

    def profile(self, enable: bool):
        _check("emb_profile", _lib.emb_profile(self._h, 1 if enable else 0))

    def profile_read(self) -> dict:
        """{kernel name: (total ms, launches)} for kernels launched since the last reset."""
        out = {}
        idx = 0
        name, ms, n = ctypes.c_char_p(), ctypes.c_double(), _I64()
        while _lib.emb_profile_read(self._h, idx, ctypes.byref(name), ctypes.byref(ms),
                                    ctypes.byref(n)) == EMB_OK:
            if n.value:
                out[name.value.decode()] = (ms.value, n.value)
            idx += 1
        return out

    def profile_reset(self):
        _check("emb_profile_reset", _lib.emb_profile_reset(self._h))

    def launch_count(self) -> int:
        return int(_lib.emb_launch_count(self._h))

    def set_adagrad_decay(self, rate: float, period_steps: int):
        """Adagrad Decay: accumulators discounted by `rate` per period of `period_steps`
        backward steps, applied when a row is next updated (0 steps: off)."""
        _check("emb_set_adagrad_decay", _lib.emb_set_adagrad_decay(self._h, float(rate),
                                                                   int(period_steps)))

    def set_admission(self, min_count: int):
        """Hashed tables: hold a key's updates until it has been looked up min_count times
        over all steps (0 or 1: no hold).  The first call starts the per-key counts and last
        steps that admission and eviction read."""
        _check("emb_set_admission", _lib.emb_set_admission(self._h, int(min_count)))

    def evict(self, max_idle_steps: int, min_count: int, stream=None, wait: bool = True):
        """Hashed tables: remove keys idle for more than max_idle_steps backward steps
        (max_idle_steps > 0) or looked up fewer than min_count times.  wait=True: waits and
        returns how many were removed; wait=False: only enqueues (returns None)."""
        n = _I64(0)
        _check("emb_evict", _lib.emb_evict(self._h, int(max_idle_steps), int(min_count),
                                           _stream(stream), ctypes.byref(n) if wait else None))
        return int(n.value) if wait else None

    def prefetch(self, ids, offsets, batch: int, stream=None):
        """Tiered tables: copy a later batch's uncached rows into the HBM cache, enqueued on
        `stream` (a second stream overlaps it with the current step); the next forward,
        eviction or watermark check waits for it.  ids/offsets as for forward, ready in the
        order of `stream` (e.g. stream.wait_stream after copying them on another stream)
        and kept alive until the stream has run it."""
        nnz = self._lookups(ids, offsets, batch)
        _check("emb_prefetch", _lib.emb_prefetch(self._h, _dptr(ids), _dptr(offsets), nnz, batch,
                                                 _stream(stream)))

    def set_tier_watermark(self, high: int, low: int = 0):
        """Tiered tables: after every backward step, when more than `high` cache rows are in
        use, write the longest-idle rows back until at most `low` remain (high = 0: off)."""
        _check("emb_set_tier_watermark", _lib.emb_set_tier_watermark(self._h, int(high), int(low)))

    def tier_occupancy(self) -> int:
        """Tiered tables: cache rows in use (waits for the device)."""
        n = _I64(0)
        _check("emb_tier_occupancy", _lib.emb_tier_occupancy(self._h, ctypes.byref(n)))
        return int(n.value)

    def key_stats(self, keys):
        """(lookup counts uint32, last step uint32) of hashed keys (0, 0: absent)."""
        import numpy as np
        keys = np.ascontiguousarray(keys, dtype=np.int64)
        cnt = np.empty(keys.size, np.uint32)
        last = np.empty(keys.size, np.uint32)
        _check("emb_read_key_stats", _lib.emb_read_key_stats(self._h, _hptr(keys), keys.size,
                                                             _hptr(cnt), _hptr(last)))
        return cnt, last

    def step_tracks_once(self) -> bool:
        """Whether the last forward's step updates rows looked up once in the backward."""
        return int(_lib.emb_step_tracks_once(self._h)) == 1
