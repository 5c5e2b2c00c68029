"""Shared helpers of the GPU parity tests (comparison rules and device plumbing)."""
import os

import numpy as np

TOL_F32 = 1e-5   # max relative error for fp32 tables
TOL_BF16 = 2e-2  # max relative error for bf16 tables with fp32 accumulation

# Error statistics of every compared output, per test:
# {(test id, what): [R17 ratio, plain rel. error (|ref| >= 1e-3 m), plain rel. error
#  (|ref| >= m / 2), entries, tolerance]}; the R17 ratio is max |gpu - ref| / max(|ref|, m),
# the quantity the tolerance bounds.  Printed by the terminal summary hook in conftest.py.
REL_ERR = {}


def tol_for(w) -> float:
    return TOL_BF16 if w.dtype == "bf16" else TOL_F32


def assert_close(gpu, ref, mag, tol, what=""):
    """|gpu - ref| <= tol * max(|ref|, mag), elementwise; mag is the oracle's magnitude of
    the expression (sum of absolute terms), so cancellation does not turn rounding noise
    into a relative error.  Also |gpu - ref| <= tol * |ref| wherever |ref| >= mag / 2.
    Returns the plain max relative error over entries with |ref| >= 1e-3 * mag, for
    reporting."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    mag = np.broadcast_to(np.asarray(mag, np.float64), ref.shape)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    bound = tol * np.maximum(np.abs(ref), mag)
    err = np.abs(gpu - ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} entries out of tolerance {tol}; first "
            + ", ".join(f"{tuple(i)}: gpu={gpu[tuple(i)]!r} ref={ref[tuple(i)]!r} mag={mag[tuple(i)]!r}"
                        for i in idx))
    scale = np.maximum(np.abs(ref), mag)
    ratio = float(np.max(np.where(scale > 0, err / np.where(scale > 0, scale, 1.0), 0.0))) if err.size else 0.0
    mag_pos = np.maximum(mag, 1e-300)
    sel = np.abs(ref) >= 1e-3 * mag_pos
    rel = float(np.max(err[sel] / np.abs(ref[sel]))) if sel.any() else 0.0
    sel2 = (np.abs(ref) >= 0.5 * mag_pos) & (np.abs(ref) > 0)
    rel2 = float(np.max(err[sel2] / np.abs(ref[sel2]))) if sel2.any() else 0.0
    # where the expression's terms cancel by at most half (|ref| >= m / 2) the plain relative
    # error itself is within the tolerance; below that, fp32 accumulation in any order is
    # bounded only relative to m (reading R17)
    if rel2 > tol:
        i = np.argwhere(sel2 & (err > tol * np.abs(ref)))[0]
        raise AssertionError(f"{what}: plain relative error {rel2:.3e} > {tol} where |ref| >= m/2; "
                             f"first {tuple(i)}: gpu={gpu[tuple(i)]!r} ref={ref[tuple(i)]!r} mag={mag[tuple(i)]!r}")
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    old = REL_ERR.get((test, what), [0.0, 0.0, 0.0, 0, tol])
    REL_ERR[(test, what)] = [max(old[0], ratio), max(old[1], rel), max(old[2], rel2),
                             old[3] + int(err.size), tol]
    return rel


def to_dev(a, torch):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def global_to_local(base, keys):
    """Global row numbers -> (table, table-local id)."""
    keys = np.asarray(keys, np.int64)
    t = np.searchsorted(base, keys, side="right") - 1
    return t, keys - base[t]


def read_gpu_rows(ctx, base, keys):
    """Rows of the GPU context for global row numbers (static tables)."""
    t, ids = global_to_local(base, keys)
    D = ctx.D
    AW = 1 if ctx.rowwise else D
    w = np.empty((len(keys), D), np.float32)
    acc = np.empty((len(keys), AW), np.float32)
    for tt in np.unique(t):
        sel = np.nonzero(t == tt)[0]
        wt, at, _ = ctx.read_rows(int(tt), ids[sel])
        w[sel], acc[sel] = wt, at
    return w, acc


def build_lib():
    """Build libemb.so through the package's build script, loaded by path so that the
    package itself (which refuses to import without the library) is not imported first."""
    import importlib.util
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    path = os.path.join(root, "recommender_model_embedding_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_emb_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()
