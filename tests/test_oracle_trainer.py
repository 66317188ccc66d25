"""Pins of the oracle's trainer update (Adam with bias correction, decoupled
weight decay and a gradient scale), against what the mathematics and an
independent library fix:
- torch.optim.AdamW / torch.optim.Adam in float64 over several steps;
- the first step from zero moments moves every parameter by lr*sign(g)
  (up to eps), whatever the betas;
- beta1 = beta2 = 0 reduces every step to p - lr*g/(|g| + eps);
- a zero gradient with zero moments only decays the parameter;
- with eps = 0 the update is invariant to scaling the gradient;
- grad_scale s on a gradient g equals scale 1 on s*g (powers of two)."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")

LR, B1, B2, EPS = 1e-3, 0.9, 0.999, 1e-8


def _rand(seed, n=1000):
    rng = np.random.default_rng(seed)
    return rng.normal(0, 1, n), rng.normal(0, 0.1, n)


@pytest.mark.parametrize("wd", [0.0, 0.01])
def test_matches_torch_adamw_float64_over_steps(wd):
    p0, _ = _rand(1)
    rng = np.random.default_rng(2)
    grads = [rng.normal(0, 0.1, p0.size) for _ in range(5)]
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([tp], lr=LR, betas=(B1, B2), eps=EPS, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    for t, g in enumerate(grads, start=1):
        tp.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = oracle.adam_update(p, g, m, v, LR, B1, B2, EPS, wd, t)
        st = opt.state[tp]
        np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-12, atol=1e-18)
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-12, atol=1e-20)


def test_matches_torch_adam_without_decay():
    p0, g = _rand(3)
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.Adam([tp], lr=LR, betas=(B1, B2), eps=EPS)
    tp.grad = torch.tensor(g, dtype=torch.float64)
    opt.step()
    p, _, _ = oracle.adam_update(p0, g, np.zeros_like(p0), np.zeros_like(p0), LR, B1, B2, EPS,
                                 0.0, 1)
    np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("betas", [(0.9, 0.999), (0.5, 0.9), (0.0, 0.0)])
def test_first_step_moves_by_lr_times_sign(betas):
    p0, g = _rand(4)
    z = np.zeros_like(p0)
    p, m, v = oracle.adam_update(p0, g, z, z, LR, betas[0], betas[1], EPS, 0.0, 1)
    np.testing.assert_allclose(p, p0 - LR * g / (np.abs(g) + EPS), rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(m, (1 - betas[0]) * g, rtol=1e-15)
    np.testing.assert_allclose(v, (1 - betas[1]) * g * g, rtol=1e-15)


def test_zero_betas_reduce_every_step_to_sign_descent():
    p0, g = _rand(5)
    rng = np.random.default_rng(6)
    m, v = rng.normal(0, 1, p0.size), rng.uniform(0, 1, p0.size)  # ignored when betas are 0
    p, m2, v2 = oracle.adam_update(p0, g, m, v, LR, 0.0, 0.0, EPS, 0.0, 7)
    np.testing.assert_allclose(p, p0 - LR * g / (np.abs(g) + EPS), rtol=1e-13, atol=1e-16)
    np.testing.assert_array_equal(m2, g)
    np.testing.assert_array_equal(v2, g * g)


def test_zero_gradient_only_decays():
    p0, _ = _rand(7)
    z = np.zeros_like(p0)
    p, m, v = oracle.adam_update(p0, z, z, z, 0.01, B1, B2, EPS, 0.1, 3)
    np.testing.assert_allclose(p, p0 * (1 - 0.01 * 0.1), rtol=1e-15)
    assert not m.any() and not v.any()


def test_eps_zero_update_is_invariant_to_gradient_scale():
    p0, g = _rand(8)
    rng = np.random.default_rng(9)
    m, v = rng.normal(0, 0.05, p0.size), rng.uniform(0.001, 0.01, p0.size)
    a, _, _ = oracle.adam_update(p0, g, m, v, LR, B1, B2, 0.0, 0.0, 4)
    b, _, _ = oracle.adam_update(p0, 3.7 * g, 3.7 * m, 3.7 ** 2 * v, LR, B1, B2, 0.0, 0.0, 4)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-16)


def test_grad_scale_is_a_multiplier_on_the_gradient():
    p0, g = _rand(10)
    z = np.zeros_like(p0)
    a = oracle.adam_update(p0, 128.0 * g, z, z, LR, B1, B2, EPS, 0.01, 2, grad_scale=1 / 128)
    b = oracle.adam_update(p0, g, z, z, LR, B1, B2, EPS, 0.01, 2)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
