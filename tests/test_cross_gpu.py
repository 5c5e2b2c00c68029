"""Cross interaction layer (reading R22: out = x0 * (xl . w) + b + xl per sample) against
the oracle, forward and backward, within the fp32 tolerance relative to the magnitude of
each expression."""
import numpy as np
import pytest

import oracle
from helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from helpers import build_lib
    build_lib()
    import recommender_model_embedding_gb300 as E
    return E


def _inputs(B, K, seed):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    return f(B, K), f(B, K), (f(K) / np.sqrt(K)).astype(np.float32), f(K), f(B, K)


def _run(E, x0, xl, w, b, dout):
    import torch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    B, K = x0.shape
    out = torch.empty((B, K), device="cuda")
    E.cross_forward(t(x0), t(xl), t(w), t(b), out)
    dx0, dxl = torch.empty((B, K), device="cuda"), torch.empty((B, K), device="cuda")
    dw, db = torch.full((K,), 7.0, device="cuda"), torch.full((K,), 7.0, device="cuda")
    E.cross_backward(t(x0), t(xl), t(w), t(dout), dx0, dxl, dw, db)
    torch.cuda.synchronize()
    return [a.cpu().numpy() for a in (out, dx0, dxl, dw, db)]


def _check(E, B, K, seed, tol=1e-5):
    x0, xl, w, b, dout = _inputs(B, K, seed)
    out, dx0, dxl, dw, db = _run(E, x0, xl, w, b, dout)
    ro, mo = oracle.cross_forward(x0, xl, w, b)
    assert_close(out, ro, mo, tol, "cross out")
    (r0, rl, rw, rb), (m0, ml, mw, mb) = oracle.cross_backward(x0, xl, w, dout)
    assert_close(dx0, r0, m0, tol, "dx0")
    assert_close(dxl, rl, ml, tol, "dxl")
    assert_close(dw, rw, mw, tol, "dw")
    assert_close(db, rb, mb, tol, "db")


@pytest.mark.parametrize("K", [4, 128, 3456, 9216, 6, 1, 130])
@pytest.mark.parametrize("B", [1, 7, 300])
def test_cross_matches_oracle(E, B, K):
    """Widths on the 16-byte path (multiples of 4, up to the maximum) and on the scalar path,
    with ragged batch sizes."""
    _check(E, B, K, seed=B * 100000 + K)


def test_cross_full_size(E):
    """The Criteo-shaped batch: 65536 samples of 27 x 128 concatenated features."""
    _check(E, 65536, 27 * 128, seed=5)


def test_cross_empty_batch_and_bad_width(E):
    import torch
    K = 8
    dw, db = torch.full((K,), 3.0, device="cuda"), torch.full((K,), 3.0, device="cuda")
    z = torch.empty((0, K), device="cuda")
    E.cross_backward(z, z, torch.zeros(K, device="cuda"), z, z, z, dw, db)
    torch.cuda.synchronize()
    assert not dw.any() and not db.any()
    big = torch.empty((1, E.CROSS_MAX_K + 4), device="cuda")
    wb = torch.empty(E.CROSS_MAX_K + 4, device="cuda")
    with pytest.raises(E.EmbError):
        E.cross_forward(big, big, wb, wb, big)
