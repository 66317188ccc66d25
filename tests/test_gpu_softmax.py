"""GPU parity: masked attention softmax forward and backward against the FP64
oracle, through the C ABI.

Every output is held to the element-wise tolerance and to the scale-aware
bounds of tests/softmax_checks.py (row sums, exact zeros, non-zero valid
entries).

The full layer tensors run on the GPU in one call (the launch the benchmark
times) and are compared on every element, a chunk of batch elements at a time.  The
shape sweep (k_len 16..4096, 2^22 elements, random valid length per row) is
checked on every element; so are rows longer than 16384 keys (the two-pass
online path, up to 2^20 keys).  The backward is checked on identical explicit
inputs (the oracle's y rounded to storage; the GPU forward's own y) and, for
the chain, against the oracle's forward-then-backward."""
import numpy as np
import pytest

import oracle
from transformer_layer_non_gb300 import ls_ops, synth
from tests.gpu_util import Guarded, assert_close, dev, f64, require_gpu, tdtype
from tests.softmax_checks import batch_chunks, check_grad, check_probs, valid_mask

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


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


def compare_all(x, dy, key_len, causal, y_t, dx_chain_t, what):
    """Every element, a chunk of batch elements at a time.  Forward: GPU y vs the
    oracle.  Backward: (a) the GPU backward of the oracle's y rounded to
    storage vs the oracle backward of that same y; (b) the chained GPU
    forward->backward vs the oracle backward of the GPU's own y (identical
    inputs) and vs the oracle's forward->backward."""
    y_gpu = f64(y_t)
    dx_chain = f64(dx_chain_t)
    ys16 = np.empty_like(x)
    refs = []
    chunks = batch_chunks(x.shape)
    for sl in chunks:
        b = f"{sl.start}:{sl.stop}"
        kl = None if key_len is None else key_len[sl]
        valid = valid_mask(x[sl].shape, kl, causal)
        ry = oracle.softmax_fwd(x[sl], kl, causal)
        check_probs(y_gpu[sl], ry, valid, x.dtype, f"{what} [b={b}]")
        yg = y_gpu[sl]
        check_grad(dx_chain[sl], oracle.softmax_bwd(yg, dy[sl], kl, causal), yg,
                   dy[sl].astype(np.float64), valid, x.dtype, f"{what} chained [b={b}]")
        assert_close(dx_chain[sl], oracle.softmax_bwd(ry, dy[sl], kl, causal),
                     f"{what} oracle chain dx [b={b}]")
        ys16[sl] = ry.astype(x.dtype)
        refs.append(valid)
    dx_a = f64(run_bwd(dev(ys16), dy, key_len, causal))
    for sl, valid in zip(chunks, refs):
        kl = None if key_len is None else key_len[sl]
        y_in = ys16[sl].astype(np.float64)
        check_grad(dx_a[sl], oracle.softmax_bwd(y_in, dy[sl], kl, causal), y_in,
                   dy[sl].astype(np.float64), valid, x.dtype,
                   f"{what} explicit [b={sl.start}:{sl.stop}]")


@pytest.mark.parametrize("name", ["tiny", "transformer-base", "bert-base", "gpt2-large"])
def test_layer_configs_every_element(name):
    require_gpu()
    L = synth.LAYERS[name]
    d = synth.layer_inputs(L, 0, which={"scores", "scores_dy", "key_len"})
    x, dy, kl = d["scores"], d["scores_dy"], d.get("key_len")
    y = run_fwd(x, kl, L.causal)
    dx = run_bwd(y, dy, kl, L.causal)
    compare_all(x, dy, kl, L.causal, y, dx, name)


@pytest.mark.parametrize("k_len", synth.SWEEP_K_LENS)
def test_sweep_every_element(k_len):
    require_gpu()
    x, dy, kl = synth.sweep_inputs(k_len)
    y_t = run_fwd(x, kl, False)
    dx_t = run_bwd(y_t, dy, kl, False)
    compare_all(x, dy, kl, False, y_t, dx_t, f"sweep {k_len}")


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
    compare_all(x, dy, kl, causal, y, dx, f"{dtype} {shape}")


def test_no_mask_and_in_place():
    require_gpu()
    x = synth.normal(10, "smi/x", (2, 4, 16, 512), 0.0, 3.0, "f16")
    dy = synth.normal(10, "smi/dy", (2, 4, 16, 512), 0.0, 1.0, "f16")
    ry = oracle.softmax_fwd(x)
    y = run_fwd(x, None, False, in_place=True)
    valid = np.ones(x.shape, dtype=bool)
    check_probs(f64(y), ry, valid, x.dtype, "in-place")
    y16 = ry.astype(np.float16)
    dyt = dev(dy)
    ls_ops.ls_softmax_bwd(dyt, dev(y16), dyt)  # dx over dy
    torch.cuda.synchronize()
    yin = y16.astype(np.float64)
    check_grad(f64(dyt), oracle.softmax_bwd(y16, dy), yin, dy.astype(np.float64), valid,
               x.dtype, "in-place")


def test_long_rows_in_place():
    # Rows past the on-chip limit are read twice; in place, the second pass
    # must still see the inputs (each thread rewrites only what it reads).
    require_gpu()
    shape = (1, 2, 2, 32768)
    x = synth.normal(11, "sml/x", shape, 0.0, 3.0, "f16")
    dy = synth.normal(11, "sml/dy", shape, 0.0, 1.0, "f16")
    kl = np.array([20001], dtype=np.int32)
    valid = valid_mask(shape, kl, True)
    ry = oracle.softmax_fwd(x, kl, True)
    y = run_fwd(x, kl, True, in_place=True)
    check_probs(f64(y), ry, valid, x.dtype, "long in-place")
    y16 = ry.astype(np.float16)
    dyt = dev(dy)
    ls_ops.ls_softmax_bwd(dyt, dev(y16), dyt, dev(kl), True)
    torch.cuda.synchronize()
    yin = y16.astype(np.float64)
    check_grad(f64(dyt), oracle.softmax_bwd(y16, dy, kl, True), yin, dy.astype(np.float64),
               valid, x.dtype, "long in-place")


def test_no_device_side_failures_after_streamed_rows():
    # The warp-per-row softmax streams rows through shared memory with bulk
    # copies and bounded waits; none of the calls above may have timed out.
    require_gpu()
    x, dy, kl = synth.sweep_inputs(512)
    y = run_fwd(x, kl, False)
    run_bwd(y, dy, kl, False)
    assert ls_ops.check_device_errors() == 0
