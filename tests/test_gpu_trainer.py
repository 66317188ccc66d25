"""GPU parity: the fused trainer update (Adam with bias correction, decoupled
weight decay and a gradient scale over one flat workspace) against the FP64
oracle, through the C ABI.

Each step feeds the GPU's own state from the previous step to both sides, so
every step is checked on its own: parameters (FP16 or FP32 storage) within
|err| <= 2e-3 + 2e-3*|ref|, the FP32 moments within 1e-5 relative.  Sizes
cover the scalar tail (n % 8), several vectors, and the BERT-base workspace
(109,482,240 values, checked on sampled elements)."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_close, require_gpu
from transformer_layer_non_gb300 import ls_ops, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LR, B1, B2, EPS = 1e-3, 0.9, 0.999, 1e-8


def f32(x):
    return float(np.float32(x))


def _check(before, after, idx, hp, step, what):
    p0, g0, m0, v0 = (t[idx].double().cpu().numpy() if idx is not None
                      else t.double().cpu().numpy() for t in before)
    p1, m1, v1 = (t[idx].double().cpu().numpy() if idx is not None
                  else t.double().cpu().numpy() for t in after)
    rp, rm, rv = oracle.adam_update(p0, g0, m0, v0, f32(hp["lr"]), f32(hp["b1"]), f32(hp["b2"]),
                                    f32(hp["eps"]), f32(hp["wd"]), step, f32(hp["gs"]))
    assert_close(p1, rp, f"{what} param")
    # The tolerance above is as large as one update (lr = 1e-3), so also hold
    # the parameters to their storage rounding: within one unit in the last
    # place of the storage dtype of the FP64 result, plus the FP32 arithmetic
    # error, which scales with the terms (old parameter and update) rather than
    # with their difference.
    if after[0].dtype == torch.float16:
        ulp = np.spacing(np.abs(rp).astype(np.float16)).astype(np.float64)
    else:
        ulp = np.spacing(np.abs(rp).astype(np.float32)).astype(np.float64)
    bad = np.abs(p1 - rp) > ulp + 1e-6 * (np.abs(p0) + np.abs(rp - p0)) + 1e-12
    assert not bad.any(), f"{what} param: {bad.sum()} elements off by more than one ulp"
    np.testing.assert_allclose(m1, rm, rtol=1e-5, atol=1e-10, err_msg=f"{what} exp_avg")
    np.testing.assert_allclose(v1, rv, rtol=1e-5, atol=1e-14, err_msg=f"{what} exp_avg_sq")


def _run_steps(n, dtype, hp, steps=(1, 2, 3), sample=None):
    p, g, m, v = synth.trainer_state(n, seed=n % 97, dtype=dtype, device="cuda")
    idx = None
    if sample is not None:
        rng = np.random.default_rng(n)
        idx = torch.from_numpy(np.unique(np.concatenate([
            rng.integers(0, n, sample), np.arange(min(n, 16)), np.arange(max(0, n - 16), n)])
        )).cuda()
    for t in steps:
        before = [x.clone() for x in (p, g, m, v)]
        ls_ops.ls_adam_update(p, g, m, v, hp["lr"], hp["b1"], hp["b2"], hp["eps"], hp["wd"], t,
                              hp["gs"])
        torch.cuda.synchronize()
        _check(before, (p, m, v), idx, hp, t, f"{dtype} n={n} step {t}")
        g.copy_(torch.roll(g, 1))  # a different gradient for the next step


HP = dict(lr=LR, b1=B1, b2=B2, eps=EPS, wd=0.01, gs=1.0)


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 65543])
def test_small_and_ragged(dtype, n):
    require_gpu()
    _run_steps(n, dtype, HP)


def test_loss_scaled_gradients_and_zero_betas():
    require_gpu()
    # Gradients stored 1024x larger (a loss scale), unscaled by grad_scale.
    _run_steps(100003, "f16", dict(HP, gs=1.0 / 1024))
    # beta1 = beta2 = 0: sign descent, bias corrections of 1.
    _run_steps(4099, "f16", dict(HP, b1=0.0, b2=0.0, wd=0.0), steps=(1, 5))


def test_bert_base_workspace_sampled():
    require_gpu()
    _run_steps(synth.TRAINER_N, "f16", HP, steps=(1, 10), sample=200000)


def test_zero_length_is_a_no_op():
    require_gpu()
    e = torch.empty(0, dtype=torch.float16, device="cuda")
    f = torch.empty(0, dtype=torch.float32, device="cuda")
    ls_ops.ls_adam_update(e, e.clone(), f, f.clone(), LR, B1, B2, EPS, 0.0, 1)
    torch.cuda.synchronize()
