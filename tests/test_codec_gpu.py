"""int8 row codec against the oracle (reading R21: per-row absmax scale / 127, codes rounded
to nearest even and clamped to +-127, decode = code * scale, all in fp32).  Codes, scales
and decoded rows must match bit for bit."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from helpers import build_lib
    build_lib()
    import recommender_model_embedding_gb300 as E
    return E


def _roundtrip(E, x):
    import torch
    n, d = x.shape
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    q = torch.empty((n, d), dtype=torch.int8, device="cuda")
    s = torch.empty(n, dtype=torch.float32, device="cuda")
    E.quantize_rows(xd, q, s)
    y = torch.empty((n, d), dtype=torch.float32, device="cuda")
    E.dequantize_rows(q, s, y)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy(), y.cpu().numpy()


def _check(E, x):
    q, s, y = _roundtrip(E, x)
    oq, os_, _ = *oracle.quantize_rows(x), None
    np.testing.assert_array_equal(s.view(np.uint32), os_.view(np.uint32))
    np.testing.assert_array_equal(q, oq)
    oy = oracle.dequantize_rows(oq, os_)
    np.testing.assert_array_equal(y.view(np.uint32), oy.view(np.uint32))


@pytest.mark.parametrize("d", [4, 16, 32, 64, 128, 132, 512, 1024, 6, 1, 1030])
@pytest.mark.parametrize("n", [1, 7, 1001])
def test_codec_matches_oracle(E, n, d):
    """Widths on the 16-byte path (multiples of 4 up to 1024 floats: one to eight chunks per
    lane) and on the scalar path (6, 1, 1030), with ragged row counts."""
    rng = np.random.default_rng(n * 10000 + d)
    x = (rng.standard_normal((n, d)) * rng.uniform(1e-3, 1e3, size=(n, 1))).astype(np.float32)
    _check(E, x)


def test_codec_special_rows(E):
    """Zero rows, rows whose quotients are exact ties, denormal and huge magnitudes."""
    d = 8
    rows = [np.zeros(d),
            [127.0, 62.5, -3.5, 0.49, -127.0, 2.5, 0.5, -0.5],
            [0.75, 1.25, -63.5, 0.0, 63.5, -0.25, 0.25, 1.75],
            np.full(d, 1e-40), [1e-45, -1e-45, 0, 0, 0, 0, 0, 0],
            np.linspace(-3e38, 3e38, d)]
    _check(E, np.array(rows, np.float32))


def test_codec_full_size_pooled_rows(E):
    """The Criteo-shaped pooled tensor of one batch (65536 x 26 rows of 128), element by
    element."""
    import torch
    w = synth.workload(2)
    rng = np.random.default_rng(22)
    x = (rng.standard_normal((w.batch * w.num_tables, w.dim)) * 0.05).astype(np.float32)
    _check(E, x)


def test_codec_empty_and_bad_arguments(E):
    import torch
    z = torch.empty((0, 8), device="cuda")
    E.quantize_rows(z, torch.empty((0, 8), dtype=torch.int8, device="cuda"),
                    torch.empty(0, device="cuda"))
    with pytest.raises(E.EmbError):
        E.quantize_rows(torch.empty((2, 0), device="cuda"),
                        torch.empty((2, 0), dtype=torch.int8, device="cuda"),
                        torch.empty(2, device="cuda"))
