"""GPU parity: cross entropy over vocabulary rows, forward (loss and lse,
FP32) and backward (logit gradients in the storage dtype), against the FP64
oracle through the C ABI, |err| <= 2e-3 + 2e-3*|ref|.  Rows are independent,
so the full-size launches (BERT-base and GPT-2-large vocabularies padded to a
multiple of 8) are checked on sampled rows; small cases on every element.
Covers label smoothing, ignored and out-of-range targets, an upstream
gradient or none, FP16/FP32 and the in-place backward."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import Guarded, assert_close, dev, f64, require_gpu, tdtype
from transformer_layer_non_gb300 import ls_ops, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _inputs(rows, V, dtype, seed):
    z = synth.normal(seed, f"ce{rows}x{V}/z", (rows, V), 0.0, 2.0, dtype)
    rng = np.random.default_rng(seed)
    t = rng.integers(0, V, rows).astype(np.int32)
    t[::7] = -100            # ignored
    if rows > 3:
        t[3] = V + 5         # out of range: ignored too
    g = rng.normal(1.0, 0.5, rows)
    return z, t, g


def _run(rows, V, dtype, eps, sample=None, seed=0):
    z, t, g = _inputs(rows, V, dtype, seed)
    zt, tt = dev(z), dev(t)
    loss = Guarded((rows,), torch.float32)
    lse = Guarded((rows,), torch.float32)
    ls_ops.ls_cross_entropy_fwd(loss.t, lse.t, zt, tt, eps, -100)
    dz = Guarded((rows, V), tdtype(z.dtype))
    gt = dev(g.astype(np.float32))
    ls_ops.ls_cross_entropy_bwd(dz.t, zt, tt, lse.t, gt, eps, -100)
    torch.cuda.synchronize()
    for b in (loss, lse, dz):
        b.check()
    idx = np.arange(rows) if sample is None else np.unique(
        np.concatenate([np.random.default_rng(seed).integers(0, rows, sample), [0, 3, rows - 1]]))
    rl, rlse = oracle.cross_entropy_fwd(z[idx], t[idx], float(np.float32(eps)), -100)
    what = f"{dtype} {rows}x{V} eps={eps}"
    assert_close(f64(loss.t)[idx], rl, f"{what} loss")
    assert_close(f64(lse.t)[idx], rlse, f"{what} lse")
    rdz = oracle.cross_entropy_bwd(z[idx], t[idx], g.astype(np.float32)[idx],
                                   float(np.float32(eps)), -100)
    got = f64(dz.t)[idx]
    assert_close(got, rdz, f"{what} dlogits")
    # Most gradients are about 1/vocab, far below the absolute tolerance, so
    # also hold them to the storage rounding (FP16: half an ulp, subnormals
    # included; FP32: a few ulps of FP32 arithmetic).
    if z.dtype == np.float16:
        tight = np.abs(got - rdz) <= 6e-8 + 2e-3 * np.abs(rdz)
    else:
        tight = np.abs(got - rdz) <= 1e-9 + 1e-5 * np.abs(rdz)
    assert tight.all(), f"{what} dlogits: {(~tight).sum()} values off at their own scale"
    return z, t, zt, tt, lse.t


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("rows,V", [(1, 8), (9, 48), (33, 1000), (64, 4104)])
@pytest.mark.parametrize("eps", [0.0, 0.1])
def test_small_every_element(dtype, rows, V, eps):
    require_gpu()
    _run(rows, V, dtype, eps)


@pytest.mark.parametrize("V", [30528, 50264])
def test_full_vocabularies_sampled_rows(V):
    require_gpu()
    _run(4096, V, "f16", 0.1, sample=200)


def test_in_place_backward_without_upstream_gradient():
    require_gpu()
    z, t, zt, tt, lse = _run(40, 2048, "f16", 0.0)
    ls_ops.ls_cross_entropy_bwd(zt, zt, tt, lse, None, 0.0, -100)
    torch.cuda.synchronize()
    assert_close(f64(zt), oracle.cross_entropy_bwd(z, t, None, 0.0, -100), "in-place dlogits")
