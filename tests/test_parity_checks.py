"""The softmax parity checks bind where the element-wise tolerance alone does
not.  Each case plants a plausible kernel mistake in a copy of the oracle's
output, on the CPU (nothing here runs the CUDA library): the element-wise
tolerance |err| <= 2e-3 + 2e-3*|ref| misses nearly all of it, because most
probabilities of a row of 512 keys with scores ~ N(0, 3) are far below 2e-3;
the checks of tests/softmax_checks.py reject each one.  (The tolerance flags
under a fifth of the altered entries: only those that happen to be large.)  The unaltered outputs,
rounded to FP16 as the GPU stores them, pass."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import ATOL, RTOL
from tests.softmax_checks import check_grad, check_probs, valid_mask
from transformer_layer_non_gb300 import synth

SHAPE = (2, 3, 8, 512)
KEY_LEN = np.array([300, 512], dtype=np.int32)


@pytest.fixture(scope="module")
def case(oracle_lib):
    x = synth.normal(5, "pc/x", SHAPE, 0.0, 3.0, "f16")
    dy = synth.normal(5, "pc/dy", SHAPE, 0.0, 1.0, "f16")
    valid = valid_mask(SHAPE, KEY_LEN, False)
    ry = oracle.softmax_fwd(x, KEY_LEN, False)
    y16 = ry.astype(np.float16).astype(np.float64)  # what a correct kernel stores
    rdx = oracle.softmax_bwd(y16, dy, KEY_LEN, False)
    return x, dy.astype(np.float64), valid, ry, y16, rdx


def _last_valid(valid, k):
    """Mask of the last k valid entries of every row."""
    n = valid.sum(-1, keepdims=True)
    j = np.arange(valid.shape[-1])
    return valid & (j >= n - k)


def _floor_misses_most(bad, good, ref):
    """The element-wise tolerance flags under a fifth of the entries changed."""
    altered = bad != good
    assert altered.any()
    flagged = np.abs(bad - ref) > ATOL + RTOL * np.abs(ref)
    assert flagged[altered].mean() < 0.2, flagged[altered].mean()


def _plants(valid, y):
    p = {}
    a = y.copy()
    a[_last_valid(valid, 8)] = 0.0             # the last valid vector of a row dropped
    p["dropped tail vector"] = a
    a = y.copy()
    t = _last_valid(valid, 16)
    a[t] *= 1.5                                # the tail scaled wrongly
    p["mis-scaled tail"] = a
    a = y.copy()
    a[..., 5] = np.where(valid[..., 5], 0.0, a[..., 5])   # one valid entry zeroed per row
    p["zeroed valid entry"] = a
    p["mis-normalised rows"] = y * (1.0 + 2.0 ** -8)
    return p


@pytest.mark.parametrize("mistake", ["dropped tail vector", "mis-scaled tail",
                                     "zeroed valid entry", "mis-normalised rows"])
def test_forward_mistakes_pass_the_tolerance_but_fail_the_checks(case, mistake):
    x, dy, valid, ry, y16, _ = case
    bad = _plants(valid, y16)[mistake]
    _floor_misses_most(bad, y16, ry)
    with pytest.raises(AssertionError):
        check_probs(bad, ry, valid, np.float16, "planted")


def test_masked_entry_not_exactly_zero_fails(case):
    x, dy, valid, ry, y16, _ = case
    bad = y16.copy()
    bad[0, 0, 0, 400] = 6e-8                         # a masked entry (key_len 300)
    assert not valid[0, 0, 0, 400]
    with pytest.raises(AssertionError):
        check_probs(bad, ry, valid, np.float16, "planted")


def test_backward_mistakes_fail_the_checks(case):
    x, dy, valid, ry, y16, rdx = case
    s = np.where(valid, y16 * dy, 0.0).sum(-1, keepdims=True)
    # <y, dy> taken 0.1% too large: a mis-scaled reduction
    bad = np.where(valid, y16 * (dy - s * 1.001), 0.0)
    _floor_misses_most(bad, rdx, rdx)
    with pytest.raises(AssertionError):
        check_grad(bad, rdx, y16, dy, valid, np.float16, "planted dx")
    # the last valid vector's gradient dropped
    bad = rdx.copy()
    bad[_last_valid(valid, 8)] = 0.0
    _floor_misses_most(bad, rdx, rdx)
    with pytest.raises(AssertionError):
        check_grad(bad, rdx, y16, dy, valid, np.float16, "planted dx")


def test_correct_outputs_pass(case):
    x, dy, valid, ry, y16, rdx = case
    check_probs(y16, ry, valid, np.float16, "fp16-rounded oracle")
    # a gradient computed in FP32 from the same inputs, rounded to FP16
    y32, dy32 = y16.astype(np.float32), dy.astype(np.float32)
    s32 = np.where(valid, y32 * dy32, np.float32(0)).sum(-1, keepdims=True, dtype=np.float32)
    dx32 = np.where(valid, y32 * (dy32 - s32), np.float32(0))
    check_grad(dx32.astype(np.float16).astype(np.float64), rdx, y16, dy, valid, np.float16,
               "fp32 gradient")
