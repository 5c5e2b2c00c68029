"""The Python binding checks the dtype and size of every buffer against the call's layout
before a pointer reaches the library (which trusts its caller's buffers).  No GPU is needed:
a stand-in object reports itself as a contiguous CUDA tensor, and every rejection is a
ValueError raised while the call's arguments are being prepared, before the library runs."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def E():
    from helpers import build_lib
    build_lib()
    import recommender_model_embedding_gb300 as E
    return E


class FakeCuda:
    """Shape, dtype and size of a CUDA tensor, without one."""

    def __init__(self, dtype, numel):
        import torch
        self.dtype = getattr(torch, dtype)
        self._n = numel
        self.is_cuda = True

    def is_contiguous(self):
        return True

    def numel(self):
        return self._n

    def data_ptr(self):
        # valid arguments before the bad one may have their pointer taken; the library call
        # comes only after every argument has been checked, so a ValueError means it never ran
        return 0x1000


def _ctx(E, T=2, D=16):
    ctx = object.__new__(E.EmbCtx)  # no library context: every check must fire first
    ctx._h = None
    ctx.T, ctx.D, ctx.F = T, D, T + 1
    ctx.out_width = D + (T + 1) * T // 2
    ctx.rowwise = False
    ctx._last = ("", 0)
    return ctx


def test_dptr_rejects_wrong_dtype_and_short_buffers(E):
    with pytest.raises(ValueError, match="dtype int64"):
        E._dptr(FakeCuda("int32", 8), "i64", 8, "ids")
    with pytest.raises(ValueError, match="at least 9"):
        E._dptr(FakeCuda("float32", 8), "f32", 9, "pooled")
    with pytest.raises(ValueError, match="CUDA"):
        import torch
        E._dptr(torch.zeros(4), "f32", 4, "x")


def test_hptr_rejects_wrong_dtype_and_short_arrays(E):
    with pytest.raises(ValueError, match="dtype int64"):
        E._hptr(np.zeros(8, np.int32), "i64", 8, "ids")
    with pytest.raises(ValueError, match="at least 9"):
        E._hptr(np.zeros(8, np.float32), "f32", 9, "dense")
    assert E._hptr(np.zeros(8, np.float32), "f32", 8, "dense") != 0


def test_forward_checks_ids_offsets_and_output(E):
    ctx = _ctx(E)
    with pytest.raises(ValueError, match="ids"):  # int32 ids
        ctx.forward(FakeCuda("int32", 8), None, 4, FakeCuda("float32", 4 * 2 * 16))
    with pytest.raises(ValueError, match="one-hot batch"):  # nnz != B*T without offsets
        ctx.forward(FakeCuda("int64", 7), None, 4, FakeCuda("float32", 4 * 2 * 16))
    with pytest.raises(ValueError, match="offsets"):  # offsets shorter than B*T+1
        ctx.forward(FakeCuda("int64", 20), FakeCuda("int32", 8), 4, FakeCuda("float32", 4 * 2 * 16))
    with pytest.raises(ValueError, match="pooled"):  # pooled shorter than B*T*D
        ctx.forward(FakeCuda("int64", 8), None, 4, FakeCuda("float32", 4 * 2 * 16 - 1))


def test_interaction_calls_check_every_buffer(E):
    ctx = _ctx(E)
    B, D, TD, W = 4, 16, 2 * 16, ctx.out_width
    good = lambda n: FakeCuda("float32", n)
    with pytest.raises(ValueError, match="out"):
        ctx.interact(good(B * D), good(B * TD), B, good(B * W - 1))
    with pytest.raises(ValueError, match="dense"):
        ctx.forward_interact(FakeCuda("int64", B * 2), None, B, good(B * D - 1), good(B * W))
    with pytest.raises(ValueError, match="dpooled"):
        ctx.interact_backward(good(B * W), good(B * D), good(B * TD), B, good(B * D), good(B * TD - 1))


def test_backwards_size_their_gradients_from_the_last_forward(E):
    ctx = _ctx(E)
    ctx._last = ("forward", 4)
    with pytest.raises(ValueError, match="dpooled"):
        ctx.backward_adagrad(FakeCuda("float32", 4 * 2 * 16 - 1))
    ctx._last = ("forward_interact", 4)
    with pytest.raises(ValueError, match="dout"):
        ctx.backward_interact_adagrad(FakeCuda("float32", 4 * ctx.out_width - 1),
                                      FakeCuda("float32", 64), FakeCuda("float32", 64))


def test_context_free_calls_check_their_buffers(E):
    n, d = 4, 8
    with pytest.raises(ValueError, match="q"):
        x = FakeCuda("float32", n * d)
        x.shape = (n, d)
        E.quantize_rows(x, FakeCuda("float32", n * d), FakeCuda("float32", n))  # codes not int8
    with pytest.raises(ValueError, match="inverse"):
        k = FakeCuda("int64", 10)
        E.unique_keys_noalloc(k, FakeCuda("int64", 10), FakeCuda("int64", 10), FakeCuda("int32", 1))


def test_host_step_checks_host_buffers(E):
    ctx = _ctx(E)
    B, W = 4, ctx.out_width
    f = lambda n: np.zeros(n, np.float32)
    with pytest.raises(ValueError, match="ids"):
        ctx.train_step_host(np.zeros(8, np.int32), None, B, f(B * 16), f(B * W), f(B * W), f(B * 16))
    with pytest.raises(ValueError, match="out"):
        ctx.train_step_host(np.zeros(8, np.int64), None, B, f(B * 16), f(B * W), f(B * W - 1), f(B * 16))


def test_prefetch_checks_ids_and_offsets(E):
    ctx = _ctx(E)
    with pytest.raises(ValueError, match="ids"):  # int32 ids
        ctx.prefetch(FakeCuda("int32", 8), None, 4)
    with pytest.raises(ValueError, match="one-hot batch"):  # nnz != B*T without offsets
        ctx.prefetch(FakeCuda("int64", 7), None, 4)
    with pytest.raises(ValueError, match="offsets"):  # offsets shorter than B*T+1
        ctx.prefetch(FakeCuda("int64", 20), FakeCuda("int32", 8), 4)
