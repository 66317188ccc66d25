"""GPU parity: softmax with fused dropout on the attention probabilities
against the FP64 oracle, every element, through the C ABI.  The dropout bits
must match bit for bit (keep on valid entries, 0 on masked ones); y, y_drop
and the backward within |err| <= 2e-3 + 2e-3*|ref| and within the
scale-aware bounds of tests/softmax_checks.py (y: row sums, exact zeros,
non-zero valid entries; y_drop: one storage ulp at its own scale, zero exactly
where the bit is 0; dx: the FP32 summation bound of <y, g>, g the gradient of
y).  Cases cover every row-length class of the dispatch (sub-warp, warp and
CTA per row, and the two-pass rows longer than 16384 keys), padding and causal
masks, FP16 and FP32, and the BERT-base and GPT-2-large layers at full size,
compared a chunk of batch elements at a time."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import Guarded, assert_close, assert_scaled, dev, f64, require_gpu, tdtype
from tests.softmax_checks import batch_chunks, check_grad, check_probs, valid_mask
from transformer_layer_non_gb300 import ls_ops, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

P, SEED, OFF = 0.1, 0x1234_5678_9ABC, 21


def _words(t):
    return t.cpu().numpy().view(np.uint32)


def _bits(words, shape):
    """Per-element dropout bits of the flat index, as an array of `shape`."""
    n = int(np.prod(shape))
    i = np.arange(n, dtype=np.int64)
    return ((words[i >> 5] >> (i & 31).astype(np.uint32)) & 1).astype(bool).reshape(shape)


def _case(x, dy, key_len, causal, what, p=P):
    n = x.size
    kl = dev(key_len) if key_len is not None else None
    y = Guarded(x.shape, tdtype(x.dtype))
    yd = Guarded(x.shape, tdtype(x.dtype))
    m = Guarded(((n + 31) // 32,), torch.int32)
    ls_ops.ls_softmax_dropout_fwd(y.t, yd.t, m.t, dev(x), kl, causal, p, SEED, OFF)
    torch.cuda.synchronize()
    for g in (y, yd, m):
        g.check()
    ry, ryd, rw = oracle.softmax_dropout_fwd(x, key_len, causal, p, SEED, OFF)
    np.testing.assert_array_equal(_words(m.t), rw, f"{what}: dropout bits")
    bits = _bits(rw, x.shape)
    y_gpu, yd_gpu = f64(y.t), f64(yd.t)
    # Backward (a): the oracle's y rounded to storage, the same bits, both sides.
    y_in = ry.astype(x.dtype)
    dx = Guarded(x.shape, tdtype(x.dtype))
    ls_ops.ls_softmax_dropout_bwd(dx.t, dev(y_in), dev(dy), m.t, kl, causal, p)
    torch.cuda.synchronize()
    dx.check()
    dx_a = f64(dx.t)
    ref_a = oracle.softmax_dropout_bwd(y_in, dy, rw, key_len, causal, p)
    # Backward (b): chained after the GPU forward, in place over dy_drop; held to
    # the oracle backward of the GPU's own y (identical inputs) and, at the
    # element-wise tolerance, to the oracle's forward->backward.
    dyt = dev(dy)
    ls_ops.ls_softmax_dropout_bwd(dyt, y.t, dyt, m.t, kl, causal, p)
    torch.cuda.synchronize()
    dx_b = f64(dyt)
    ref_b = oracle.softmax_dropout_bwd(y_gpu, dy, rw, key_len, causal, p)
    assert_close(dx_b, oracle.softmax_dropout_bwd(ry, dy, rw, key_len, causal, p),
                 f"{what} oracle chain dx")
    scale = 1.0 / (1.0 - p)
    y_in64 = y_in.astype(np.float64)
    for sl in batch_chunks(x.shape):
        klb = None if key_len is None else key_len[sl]
        valid = valid_mask(x[sl].shape, klb, causal)
        w = f"{what} [b={sl.start}:{sl.stop}]"
        check_probs(y_gpu[sl], ry[sl], valid, x.dtype, w)
        assert_close(yd_gpu[sl], ryd[sl], f"{w} y_drop")
        assert_scaled(yd_gpu[sl], ryd[sl], x.dtype, f"{w} y_drop", ftz=x.dtype == np.float32)
        assert (yd_gpu[sl][~bits[sl]] == 0.0).all(), f"{w}: y_drop not 0 where the bit is 0"
        g = np.where(bits[sl], dy[sl].astype(np.float64) * scale, 0.0)
        check_grad(dx_a[sl], ref_a[sl], y_in64[sl], g, valid, x.dtype, f"{w} explicit")
        check_grad(dx_b[sl], ref_b[sl], y_gpu[sl], g, valid, x.dtype, f"{w} chained")


@pytest.mark.parametrize("k_len", synth.SWEEP_K_LENS)
def test_sweep_row_lengths(k_len):
    require_gpu()
    x, dy, kl = synth.sweep_inputs(k_len, seed=7, elements=1 << 20)
    _case(x, dy, kl, False, f"sweep k_len={k_len}")


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("shape,causal", [((2, 3, 5, 24), False), ((1, 2, 7, 136), True),
                                          ((2, 2, 33, 40), True), ((1, 1, 3, 2056), False),
                                          ((1, 1, 3, 65544), True), ((2, 1, 2, 16400), False),
                                          ((1, 1, 2, 1 << 20), True)])
def test_odd_shapes_and_masks(dtype, shape, causal):
    require_gpu()
    b = shape[0]
    x = synth.normal(3, f"smd/x{shape}", shape, 0.0, 3.0, dtype)
    dy = synth.normal(3, f"smd/dy{shape}", shape, 0.0, 1.0, dtype)
    kl = np.array([shape[-1] // 2 + 1, -3, shape[-1] + 5][:b], dtype=np.int32)
    _case(x, dy, kl, causal, f"{dtype} {shape} causal={causal}")
    _case(x, dy, None, causal, f"{dtype} {shape} causal={causal} no padding", p=0.5)


@pytest.mark.parametrize("name", ["tiny", "transformer-base", "bert-base", "gpt2-large"])
def test_layer_configs(name):
    require_gpu()
    L = synth.LAYERS[name]
    d = synth.layer_inputs(L, 0, which={"scores", "scores_dy", "key_len"})
    _case(d["scores"], d["scores_dy"], d.get("key_len"), L.causal, name)


def test_p_zero_keeps_every_valid_entry():
    require_gpu()
    x, dy, kl = synth.sweep_inputs(512, seed=9, elements=1 << 16)
    _case(x, dy, kl, False, "p=0", p=0.0)
