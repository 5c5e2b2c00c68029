"""The benchmark's algorithmic-bytes model (the numerators of the reported roofline
fractions) against the per-unit figures stated for the Criteo-shaped workload: fp32 rows of
128, 26 tables, 27 interaction vectors (351 pairs), one-hot lookups."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _model(U=0, once=0, B=None):
    import bench
    w = bench.workload(False, 1, 2)
    if B is not None:
        import dataclasses
        w = dataclasses.replace(w, batch=B)
    L = w.batch * w.num_tables
    return w, bench.kernel_bytes(w, U, L, once)


def test_per_sample_figures():
    # per sample, T = 26, D = 128, W = D + 351 = 479:
    # forward 4 (T D + D + W) + 16 T = 4 * 3935 + 416 = 16,156
    # backward 4 (T D + 2 D + W) + 4 T = 4 * 4063 + 104 = 16,356
    _, kb = _model(B=1)
    assert kb["fused_fwd"] == 16156
    assert kb["fused_bwd"] == 16356


def test_per_unique_row_figures():
    # per unique row reduced in the backward: one gradient row (512 bytes); the update reads
    # and clears it and reads and writes w and acc, plus 12 bytes of indices and slot
    _, k0 = _model(U=0, B=1)
    _, k1 = _model(U=1, B=1)
    assert k1["fused_bwd"] - k0["fused_bwd"] == 512
    assert k1["adagrad_from_g"] - k0["adagrad_from_g"] == 6 * 512 + 12


def test_once_rows_move_bytes_from_the_update_to_the_backward():
    # a once row: the backward reads its accumulator and writes w and acc (3 rows) instead of
    # reducing one gradient row; the update no longer touches it
    _, a = _model(U=10, once=0, B=1)
    _, b = _model(U=10, once=4, B=1)
    assert b["fused_bwd"] - a["fused_bwd"] == 4 * (3 * 512 - 512)
    assert a["adagrad_from_g"] - b["adagrad_from_g"] == 4 * (6 * 512 + 12)
