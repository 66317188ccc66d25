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


# ---------------------------------------------------------------------------
# Checks at the values' own scale.  The element-wise tolerance above has an
# absolute floor of 2e-3, larger than almost every attention probability
# (rows of hundreds of keys, scores ~ N(0, 3)), so on its own it accepts 0 or
# any value of the right order.  These helpers hold outputs to the rounding of
# their storage format instead.
# ---------------------------------------------------------------------------
def storage_ulp(ref, np_dtype):
    """Spacing of the storage format (FP16 or FP32) at |ref|; below the
    smallest normal number, the subnormal spacing."""
    mant, emin = (10, -14) if np.dtype(np_dtype) == np.float16 else (23, -126)
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** emin)))
    return np.exp2(e - mant)


def assert_scaled(got, ref, np_dtype, what="", extra=0.0, ftz=False):
    """|err| <= 2e-3*|ref| + one storage ulp at ref + extra (an array of
    per-element error terms the caller derives, e.g. an FP32 summation bound).
    ftz: the kernel's exponential flushes FP32 results below 2^-126 to zero
    (documented), so a 0 is accepted where |ref| < 2^-126."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bound = RTOL * np.abs(ref) + storage_ulp(ref, np_dtype) + extra
    bad = err > bound
    if ftz:
        bad &= ~((got == 0.0) & (np.abs(ref) < 2.0 ** -126))
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err / bound, 0.0)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} elements off at their own scale; worst at "
            f"{idx}: got {got[idx]!r} ref {ref[idx]!r} err {err[idx]:.3g} bound {bound[idx]:.3g}")


def fp32_sum_bound(n_terms, abs_sum):
    """Bound on the error of an FP32 sum of n terms in any order (recursive or
    tree summation): gamma_n * sum|terms|, gamma_n = n*u/(1 - n*u), u = 2^-24
    (Higham, "Accuracy and Stability of Numerical Algorithms", 4.2)."""
    nu = np.asarray(n_terms, dtype=np.float64) * 2.0 ** -24
    return nu / (1.0 - nu) * abs_sum
