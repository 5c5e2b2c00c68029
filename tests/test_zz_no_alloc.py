"""The allocation-free unique-keys entry point, checked against numpy and the context path.

emb_unique_keys_noalloc serves callers that may not allocate device memory (servers with a
fixed device memory budget, plug-ins handed only their buffers): its hash-set scratch is a
fixed array inside the library.  This test calls it through the C ABI twice in a row on
different batches and compares each result, exactly (integer results), with numpy's unique
keys and counts and with the unique keys and counts of emb_forward + emb_read_unique on a
hashed context.  It runs last (file name) so that a failure here does not hide the rest of
the suite, and it does not depend on earlier tests.
"""
import numpy as np
import pytest

import synth
from helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from helpers import build_lib
    build_lib()
    import recommender_model_embedding_gb300 as E
    return E


def _keys(seed, n):
    rng = np.random.default_rng(seed)
    ranks = synth.zipf_ranks(rng, 60_000, 1.1, n) - 1
    keys = synth.key_bijection(ranks, seed)
    keys[::997] = -5  # negative keys are skipped
    return keys


def test_noalloc_unique_matches_numpy_and_context_path(E):
    import torch
    n = 200_000
    for call, seed in enumerate((11, 12)):  # two calls in a row share the scratch
        keys = _keys(seed, n)
        dk = to_dev(keys, torch)
        uniq = torch.full((n,), -7, dtype=torch.int64, device="cuda")
        inv = torch.empty(n, dtype=torch.int32, device="cuda")
        nu = torch.empty(1, dtype=torch.int32, device="cuda")
        E.unique_keys_noalloc(dk, uniq, inv, nu)
        torch.cuda.synchronize()
        U = int(nu.item())
        u = uniq[:U].cpu().numpy()
        iv = inv.cpu().numpy()
        # reference: the context path on a hashed table holding the same keys
        with E.EmbCtx(1, 4, hashed=True, capacity=1 << 18, max_batch=n, max_lookups=n) as ctx:
            ctx.forward(dk, None, n, torch.empty((n, 1, 4), device="cuda"))
            assert ctx.get_status() == E.FLAG_BAD_KEY
            rk, rc = ctx.read_unique()
        order = np.argsort(u)
        ro = np.argsort(rk)
        counts = np.bincount(iv[iv >= 0], minlength=U)
        # numpy: the distinct non-negative keys and their occurrence counts
        nk, nc = np.unique(keys[keys >= 0], return_counts=True)
        np.testing.assert_array_equal(u[order], nk)
        np.testing.assert_array_equal(counts[order], nc)
        # the context path gives the same keys and counts
        np.testing.assert_array_equal(u[order], rk[ro])
        np.testing.assert_array_equal(counts[order], rc[ro].astype(np.int64))
        valid = keys >= 0
        assert np.all(iv[~valid] == -1)
        np.testing.assert_array_equal(u[iv[valid]], keys[valid])


def test_noalloc_rejects_oversize_batch(E):
    import torch
    n = E.NOALLOC_MAX_KEYS + 1
    dk = torch.zeros(n, dtype=torch.int64, device="cuda")
    with pytest.raises(E.EmbError) as ei:
        E.unique_keys_noalloc(dk, torch.empty(n, dtype=torch.int64, device="cuda"),
                              torch.empty(n, dtype=torch.int32, device="cuda"),
                              torch.empty(1, dtype=torch.int32, device="cuda"))
    assert ei.value.status == E.EMB_EINVAL
