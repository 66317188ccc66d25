"""GPU parity: masked attention softmax forward and backward against the FP64
oracle, |err| <= 2e-3 + 2e-3*|ref|; masked entries must be exactly zero.

Full layer sizes run on the GPU in one call (the launch the benchmark times);
the oracle checks every (batch, head) slice of the smaller layers and a sample
of slices of the larger ones.  The shape sweep (k_len 16..4096, 2^22 elements,
random valid length per row) is checked on every element; rows longer than
16384 keys (the two-pass online path) up to 2^18 on every element of a few
rows."""
import numpy as np
import pytest

import oracle
from transformer_layer_non_gb300 import ls_ops, synth
from tests.gpu_util import Guarded, assert_close, dev, f64, require_gpu, tdtype

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _valid(shape, key_len, causal):
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


def run_fwd(x, key_len, causal, in_place=False):
    kl = dev(key_len) if key_len is not None else None
    if in_place:
        xt = dev(x)
        ls_ops.ls_softmax_fwd(xt, xt, kl, causal)
        torch.cuda.synchronize()
        return xt
    y = Guarded(x.shape, tdtype(x.dtype))
    ls_ops.ls_softmax_fwd(y.t, dev(x), kl, causal)
    torch.cuda.synchronize()
    y.check()
    return y.t


def run_bwd(y_t, dy, key_len, causal):
    kl = dev(key_len) if key_len is not None else None
    dx = Guarded(dy.shape, tdtype(dy.dtype))
    ls_ops.ls_softmax_bwd(dx.t, y_t, dev(dy), kl, causal)
    torch.cuda.synchronize()
    dx.check()
    return dx.t


def compare_slices(x, dy, key_len, causal, y_t, dx_chain_t, slices, what):
    """Oracle on selected (b, h) slices.  Forward: GPU y vs oracle y.  Backward:
    (a) the GPU backward of the oracle's y (rounded to storage) vs the oracle
    backward of that same y; (b) the chained GPU fwd->bwd vs the oracle chain."""
    y_gpu = f64(y_t)
    dx_chain = f64(dx_chain_t)
    ys16 = np.zeros_like(x)
    refs = {}
    for (b, h) in slices:
        kl = None if key_len is None else key_len[b:b + 1]
        xs = x[b:b + 1, h:h + 1]
        ry = oracle.softmax_fwd(xs, kl, causal)
        refs[(b, h)] = ry
        assert_close(y_gpu[b:b + 1, h:h + 1], ry, f"{what} y[{b},{h}]")
        valid = _valid(xs.shape, kl, causal)
        assert (y_gpu[b:b + 1, h:h + 1][~valid] == 0.0).all(), "masked output not exactly 0"
        rdx = oracle.softmax_bwd(ry, dy[b:b + 1, h:h + 1], kl, causal)
        assert_close(dx_chain[b:b + 1, h:h + 1], rdx, f"{what} chained dx[{b},{h}]")
        assert (dx_chain[b:b + 1, h:h + 1][~valid] == 0.0).all()
        ys16[b:b + 1, h:h + 1] = ry.astype(x.dtype)
    # (a): backward on identical explicit inputs (only the checked slices matter)
    dx_a = f64(run_bwd(dev(ys16), dy, key_len, causal))
    for (b, h) in slices:
        kl = None if key_len is None else key_len[b:b + 1]
        rdx = oracle.softmax_bwd(ys16[b:b + 1, h:h + 1], dy[b:b + 1, h:h + 1], kl, causal)
        assert_close(dx_a[b:b + 1, h:h + 1], rdx, f"{what} dx[{b},{h}]")


@pytest.mark.parametrize("name", ["tiny", "transformer-base", "bert-base", "gpt2-large"])
def test_layer_configs(name):
    require_gpu()
    L = synth.LAYERS[name]
    d = synth.layer_inputs(L, 0, which={"scores", "scores_dy", "key_len"})
    x, dy, kl = d["scores"], d["scores_dy"], d.get("key_len")
    y = run_fwd(x, kl, L.causal)
    dx = run_bwd(y, dy, kl, L.causal)
    B, Hh = x.shape[:2]
    if B * Hh <= 64:
        slices = [(b, h) for b in range(B) for h in range(Hh)]
    else:
        rng = np.random.default_rng(7)
        slices = sorted({(int(rng.integers(B)), int(rng.integers(Hh))) for _ in range(12)})
        slices += [(0, 0), (B - 1, Hh - 1)]
    compare_slices(x, dy, kl, L.causal, y, dx, slices, name)


@pytest.mark.parametrize("k_len", synth.SWEEP_K_LENS)
def test_sweep_every_element(k_len):
    require_gpu()
    x, dy, kl = synth.sweep_inputs(k_len)
    y_t = run_fwd(x, kl, False)
    ry = oracle.softmax_fwd(x, kl, False)
    y = f64(y_t)
    assert_close(y, ry, f"sweep {k_len} y")
    valid = _valid(x.shape, kl, False)
    assert (y[~valid] == 0.0).all()
    y16 = ry.astype(np.float16)
    dx = f64(run_bwd(dev(y16), dy, kl, False))
    assert_close(dx, oracle.softmax_bwd(y16, dy, kl, False), f"sweep {k_len} dx")
    assert (dx[~valid] == 0.0).all()


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("shape,causal", [
    ((2, 2, 8, 8192), False), ((1, 2, 3, 16384), True), ((3, 2, 5, 24), True),
    ((2, 3, 7, 40), False), ((2, 1, 9, 264), True), ((1, 1, 300, 1032), True),
    ((2, 2, 16, 8), True), ((1, 2, 3, 16392), True), ((2, 1, 2, 65536), False),
    ((1, 1, 2, 262144), True), ((2, 1, 3, 14344), False), ((1, 1, 2, 1 << 20), False)])
def test_odd_lengths_and_masks(dtype, shape, causal):
    # k_len classes between the sweep points, q_len != k_len with the causal
    # diagonal, and key lengths that are 0, negative, 1, or past k_len.
    require_gpu()
    b = shape[0]
    x = synth.normal(9, f"smo/x{shape}", shape, 0.0, 3.0, dtype)
    dy = synth.normal(9, f"smo/dy{shape}", shape, 0.0, 1.0, dtype)
    kl = np.array([shape[3] + 5, 0, shape[3] // 2 + 1, -3, 1][:b], dtype=np.int32)
    if b == 1:
        kl = np.array([shape[3] - 3], dtype=np.int32)
    y = run_fwd(x, kl, causal)
    dx = run_bwd(y, dy, kl, causal)
    slices = [(i, h) for i in range(shape[0]) for h in range(shape[1])]
    compare_slices(x, dy, kl, causal, y, dx, slices, f"{shape}")


def test_no_mask_and_in_place():
    require_gpu()
    x = synth.normal(10, "smi/x", (2, 4, 16, 512), 0.0, 3.0, "f16")
    dy = synth.normal(10, "smi/dy", (2, 4, 16, 512), 0.0, 1.0, "f16")
    ry = oracle.softmax_fwd(x)
    y = run_fwd(x, None, False, in_place=True)
    assert_close(f64(y), ry, "in-place y")
    y16 = ry.astype(np.float16)
    dyt = dev(dy)
    ls_ops.ls_softmax_bwd(dyt, dev(y16), dyt)  # dx over dy
    torch.cuda.synchronize()
    assert_close(f64(dyt), oracle.softmax_bwd(y16, dy), "in-place dx")


def test_long_rows_in_place():
    # Rows past the on-chip limit are read twice; in place, the second pass
    # must still see the inputs (each thread rewrites only what it reads).
    require_gpu()
    shape = (1, 2, 2, 32768)
    x = synth.normal(11, "sml/x", shape, 0.0, 3.0, "f16")
    dy = synth.normal(11, "sml/dy", shape, 0.0, 1.0, "f16")
    kl = np.array([20001], dtype=np.int32)
    ry = oracle.softmax_fwd(x, kl, True)
    y = run_fwd(x, kl, True, in_place=True)
    assert_close(f64(y), ry, "long in-place y")
    y16 = ry.astype(np.float16)
    dyt = dev(dy)
    ls_ops.ls_softmax_bwd(dyt, dev(y16), dyt, dev(kl), True)
    torch.cuda.synchronize()
    assert_close(f64(dyt), oracle.softmax_bwd(y16, dy, kl, True), "long in-place dx")


def test_no_device_side_failures_after_streamed_rows():
    # The warp-per-row softmax streams rows through shared memory with bulk
    # copies and bounded waits; none of the calls above may have timed out.
    require_gpu()
    x, dy, kl = synth.sweep_inputs(512)
    y = run_fwd(x, kl, False)
    run_bwd(y, dy, kl, False)
    assert ls_ops.check_device_errors() == 0
