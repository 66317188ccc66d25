"""Helpers shared by the GPU parity tests: device transfer, guard-banded output
buffers, and the element-wise tolerance |err| <= 2e-3 + 2e-3*|ref| that FP16
and FP32 outputs and gradients must meet against the FP64 oracle."""
import numpy as np
import pytest

ATOL = 2e-3
RTOL = 2e-3
PAD = 64  # guard elements on each side of an output (128 bytes in FP16)

torch = pytest.importorskip("torch")


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def f64(t) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def tdtype(np_dtype):
    return {np.dtype(np.float16): torch.float16, np.dtype(np.float32): torch.float32}[
        np.dtype(np_dtype)]


class Guarded:
    """An output tensor with canary-filled guard bands before and after it.
    ``check()`` asserts that no byte of the guard bands changed."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) if len(shape) else 1
        self.buf = torch.empty(n + 2 * PAD, dtype=dtype, device="cuda")
        # A canary pattern that no kernel writes by accident (also fills the body).
        self.buf.view(torch.uint8).fill_(0xA5)
        self.t = self.buf[PAD:PAD + n].view(shape)
        if fill is not None:
            self.t.fill_(fill)
        self._pad = self.buf.view(torch.uint8).clone()

    def check(self):
        now = self.buf.view(torch.uint8)
        es = self.buf.element_size()
        lo, hi = PAD * es, now.numel() - PAD * es
        assert torch.equal(now[:lo], self._pad[:lo]), "guard band before the output was written"
        assert torch.equal(now[hi:], self._pad[hi:]), "guard band after the output was written"


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} elements outside tolerance; worst at {idx}: "
            f"got {got[idx]!r} ref {ref[idx]!r} err {err[idx]:.3g} bound {bound[idx]:.3g}")


def mask_words_of(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)
