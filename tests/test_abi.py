"""The C-ABI library: it loads without a GPU, exports every entry point the header declares,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "emb.h")


@pytest.fixture(scope="module")
def lib():
    from helpers import build_lib
    path = build_lib()
    return ctypes.CDLL(path)


def declared_entry_points():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(emb_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for required in ("emb_create", "emb_forward", "emb_interact", "emb_interact_backward",
                     "emb_backward_adagrad", "emb_forward_interact",
                     "emb_backward_interact_adagrad", "emb_get_status", "emb_read_rows",
                     "emb_read_unique", "emb_export_hash", "emb_destroy", "emb_status_str",
                     "emb_train_step_host"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), f"{name} declared in emb.h but not exported"


def test_status_strings(lib):
    lib.emb_status_str.restype = ctypes.c_char_p
    assert lib.emb_status_str(0) == b"ok"
    assert lib.emb_status_str(1) == b"invalid argument"
    assert lib.emb_status_str(99) == b"unknown status"


def _cfg(**kw):
    import recommender_model_embedding_gb300 as E
    rows = kw.pop("rows_list", [10, 20])
    arr = (ctypes.c_int64 * len(rows))(*rows)
    base = dict(num_tables=len(rows), dim=16, rows=ctypes.cast(arr, ctypes.POINTER(ctypes.c_int64)),
                hashed=0, capacity=0, dtype=0, pooling=0, optimizer=0, lr=0.01, eps=1e-8,
                init_acc=0.1, init_lo=-0.05, init_hi=0.05, hash_init=0.0, seed=1, max_batch=4,
                max_lookups=8)
    base.update(kw)
    c = E.EmbConfig(**base)
    c._keep = arr
    return c


@pytest.mark.parametrize("bad", [
    dict(num_tables=0), dict(dim=0), dict(dim=6), dict(dim=4, dtype=1), dict(dtype=2),
    dict(pooling=3), dict(optimizer=7), dict(max_batch=0), dict(max_lookups=0),
    dict(eps=-1.0), dict(hashed=1, capacity=1000), dict(hashed=1, capacity=1),
    dict(rows=None), dict(rows_list=[10, 0]), dict(max_lookups=1 << 31),
])
def test_create_rejects_bad_config_without_a_device(lib, bad):
    import recommender_model_embedding_gb300 as E
    cfg = _cfg(**bad)
    h = ctypes.c_void_p()
    assert E._lib.emb_create(ctypes.byref(cfg), ctypes.byref(h)) == E.EMB_EINVAL
    assert not h.value


def test_null_context_is_rejected(lib):
    import recommender_model_embedding_gb300 as E
    L = E._lib
    assert L.emb_forward(None, None, None, 0, 0, None, None) == E.EMB_EINVAL
    assert L.emb_interact(None, None, None, 0, None, None) == E.EMB_EINVAL
    assert L.emb_interact_backward(None, None, None, None, 0, None, None, None) == E.EMB_EINVAL
    assert L.emb_backward_adagrad(None, None, None) == E.EMB_EINVAL
    assert L.emb_forward_interact(None, None, None, 0, 0, None, None, None) == E.EMB_EINVAL
    assert L.emb_backward_interact_adagrad(None, None, None, None, None) == E.EMB_EINVAL
    assert L.emb_get_status(None, None, None) == E.EMB_EINVAL
    assert L.emb_read_rows(None, 0, None, 0, None, None, None) == E.EMB_EINVAL
    assert L.emb_launch_count(None) == 0
    assert L.emb_prefetch(None, None, None, 0, 0, None) == E.EMB_EINVAL
    assert L.emb_set_tier_watermark(None, 10, 5) == E.EMB_EINVAL
    assert L.emb_tier_occupancy(None, None) == E.EMB_EINVAL
    L.emb_destroy(None)


def test_binding_and_oracle_are_independent():
    pkg = os.path.join(ROOT, "recommender_model_embedding_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                code = re.sub(r"#.*|//.*", "", text)
                assert not re.search(r"import\s+oracle|from\s+oracle|liboracle|oracle\.cpp", code), \
                    f"{f} uses the oracle"
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".cpp")):
            assert "recommender_model_embedding_gb300" not in open(os.path.join(ROOT, "oracle", f)).read()


@pytest.mark.parametrize("cache,bad", [(0, {}), (1, {}), (1000, {}), (1 << 32, {}),
                                       (1024, dict(hashed=1, capacity=1024))])
def test_create_tiered_rejects_bad_cache_without_a_device(lib, cache, bad):
    """Tiered tables: the cache size must be a power of two in [2, 2^31] and the tables
    static; checked before any device call."""
    import recommender_model_embedding_gb300 as E
    cfg = _cfg(**bad)
    h = ctypes.c_void_p()
    assert E._lib.emb_create_tiered(ctypes.byref(cfg), cache, ctypes.byref(h)) == E.EMB_EINVAL
    assert not h.value


def test_new_calls_reject_bad_arguments_without_a_device(lib):
    """Admission, eviction, decay, cross layer and codec: NULL contexts, empty or oversized
    widths and negative counts are rejected on the host."""
    import recommender_model_embedding_gb300 as E
    L = E._lib
    assert L.emb_set_admission(None, 2) == E.EMB_EINVAL
    assert L.emb_evict(None, 1, 0, None, None) == E.EMB_EINVAL
    assert L.emb_read_key_stats(None, None, 0, None, None) == E.EMB_EINVAL
    assert L.emb_set_adagrad_decay(None, 0.5, 2) == E.EMB_EINVAL
    assert L.emb_step_tracks_once(None) == -1
    for K in (0, E.CROSS_MAX_K + 1):
        assert L.emb_cross_forward(None, None, None, None, 1, K, None, None) == E.EMB_EINVAL
        assert L.emb_cross_backward(None, None, None, None, 1, K, None, None, None, None,
                                    None) == E.EMB_EINVAL
    assert L.emb_cross_forward(None, None, None, None, -1, 8, None, None) == E.EMB_EINVAL
    assert L.emb_cross_forward(None, None, None, None, 2, 8, None, None) == E.EMB_EINVAL
    assert L.emb_quantize_rows(None, -1, 8, None, None, None) == E.EMB_EINVAL
    assert L.emb_quantize_rows(None, 4, 0, None, None, None) == E.EMB_EINVAL
    assert L.emb_quantize_rows(None, 4, 8, None, None, None) == E.EMB_EINVAL
    assert L.emb_dequantize_rows(None, None, 4, 8, None, None) == E.EMB_EINVAL
