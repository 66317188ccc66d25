"""Parity checks of softmax outputs and gradients against the FP64 oracle,
shared by the softmax GPU tests (and exercised on the CPU by
test_parity_checks.py, which plants mistakes in copies of oracle outputs).

Every output is held to two bounds: the element-wise tolerance
|err| <= 2e-3 + 2e-3*|ref|, and -- because that absolute floor is larger than
almost every probability of a row of hundreds of keys -- a bound at the
value's own scale: |err| <= 2e-3*|ref| + one storage ulp at ref (+ for the
backward the FP32 summation error of <y, g>, gamma_n * sum|y*g| (Higham 4.2),
times y).  Masked entries must be exactly zero, valid entries whose reference
rounds to a non-zero storage value must be non-zero, and every row with a
valid key must sum to 1 within the output rounding."""
import numpy as np

from tests.gpu_util import assert_close, assert_scaled, fp32_sum_bound


def valid_mask(shape, key_len, causal):
    b, h, lq, lk = shape
    v = np.ones(shape, dtype=bool)
    j = np.arange(lk)
    if key_len is not None:
        kl = np.clip(np.asarray(key_len, dtype=np.int64), 0, None)
        v &= (j[None, :] < kl[:, None])[:, None, None, :]
    if causal:
        q = np.arange(lq)
        v &= (j[None, :] <= (q[:, None] + lk - lq))[None, None, :, :]
    return v


def check_probs(y, ref, valid, np_dtype, what):
    """Forward outputs y (float64 view of the GPU's storage values) against the
    oracle's probabilities ref, on the entries `valid` says are valid."""
    fp16 = np.dtype(np_dtype) == np.float16
    assert_close(y, ref, f"{what} y")
    assert_scaled(y, ref, np_dtype, f"{what} y", ftz=not fp16)
    assert (y[~valid] == 0.0).all(), f"{what}: masked output not exactly 0"
    smallest = 2.0 ** -24 if fp16 else 2.0 ** -126
    need = valid & (np.abs(ref) >= smallest)
    zero = need & (y == 0.0)
    assert not zero.any(), f"{what}: {int(zero.sum())} valid entries with a non-zero reference are 0"
    nvalid = valid.sum(-1)
    sums = np.where(valid, y, 0.0).sum(-1)
    # Each output rounds by half an ulp (FP16: relative 2^-11, at most 2^-25
    # absolute for subnormals); the FP32 normaliser adds gamma_n.
    tol = ((2.0 ** -10 if fp16 else 2.0 ** -18) + nvalid * (2.0 ** -24 if fp16 else 2.0 ** -126)
           + fp32_sum_bound(nvalid, 1.0))
    off = (nvalid > 0) & (np.abs(sums - 1.0) > tol)
    assert not off.any(), (f"{what}: {int(off.sum())} rows do not sum to 1; worst "
                           f"{float(np.abs(sums - 1.0)[off].max()):.3g}")
    assert (sums[nvalid == 0] == 0.0).all(), f"{what}: a row with no valid key is not all 0"


def check_grad(dx, ref, y, g, valid, np_dtype, what):
    """Backward outputs dx against the oracle's ref = y*(g - <y, g>), computed
    from the very inputs (y, g) the GPU got: the FP32 error of <y, g> and of
    the elementwise steps enters as y*gamma_(n+3)*(|g| + sum|y*g|)."""
    assert_close(dx, ref, f"{what} dx")
    n = valid.sum(-1, keepdims=True)
    s_abs = np.where(valid, np.abs(y * g), 0.0).sum(-1, keepdims=True)
    extra = np.abs(y) * fp32_sum_bound(n + 3, np.abs(g) + s_abs)
    assert_scaled(dx, ref, np_dtype, f"{what} dx", extra=extra)
    assert (dx[~valid] == 0.0).all(), f"{what}: masked gradient not exactly 0"


def batch_chunks(shape, max_elements=1 << 22):
    """Slices of the batch axis holding about max_elements elements each (at
    least one batch element), so that checks of large tensors stay in memory
    and checks of many tiny rows stay fast."""
    per = int(np.prod(shape[1:]))
    step = max(1, max_elements // max(per, 1))
    return [slice(b, min(b + step, shape[0])) for b in range(0, shape[0], step)]
