"""Pins for the oracle's LayerNorm forward and backward.

"CMU 11-868 L10 (LightSeq)", technique 2: the statistics rewrite
sigma = sqrt(mu(x^2) - mu(x)^2) (slide p.21) and the backward pass as two
parallel sums sum_j w_j dy_j and sum_j w_j dy_j x_j plus elementwise work
(slide p.22).  The oracle itself computes the two-pass definition; these tests
tie it to a library routine (torch in float64), to finite differences, to
closed forms, and to the pages' rewritten forms.
"""
import numpy as np
import pytest
import torch

import oracle

EPS = 1e-5


@pytest.fixture
def ln_case():
    rng = np.random.default_rng(0)
    rows, cols = 5, 64
    x = rng.standard_normal((rows, cols)) * 1.7 + 0.3
    gamma = rng.normal(1.0, 0.1, cols)
    beta = rng.normal(0.0, 0.1, cols)
    dy = rng.standard_normal((rows, cols))
    return x, gamma, beta, dy


def test_fwd_matches_torch_float64(ln_case):
    x, g, b, _ = ln_case
    y, mean, rstd = oracle.layernorm_fwd(x, g, b, EPS)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (x.shape[1],), torch.from_numpy(g),
                                         torch.from_numpy(b), EPS).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-13, atol=1e-14)


def test_unit_affine_gives_zero_mean_and_closed_form_variance(ln_case):
    x, _, _, _ = ln_case
    cols = x.shape[1]
    y, mean, rstd = oracle.layernorm_fwd(x, np.ones(cols), np.zeros(cols), EPS)
    assert np.abs(y.mean(axis=1)).max() <= 1e-12
    var = ((x - x.mean(axis=1, keepdims=True)) ** 2).mean(axis=1)
    np.testing.assert_allclose(y.var(axis=1), var / (var + EPS), rtol=1e-12)
    # eps = 0 gives variance exactly 1 (to rounding).
    y0, _, _ = oracle.layernorm_fwd(x, np.ones(cols), np.zeros(cols), 0.0)
    np.testing.assert_allclose(y0.var(axis=1), 1.0, rtol=1e-12)


def test_one_pass_variance_equals_two_pass(ln_case):
    # The single-sync rewrite var = mu(x^2) - mu(x)^2 agrees with the two-pass
    # definition the oracle uses (FP64, well-conditioned rows).
    x, g, b, _ = ln_case
    _, mean, rstd = oracle.layernorm_fwd(x, g, b, EPS)
    var_two_pass = 1.0 / rstd**2 - EPS
    var_one_pass = (x**2).mean(axis=1) - x.mean(axis=1) ** 2
    np.testing.assert_allclose(var_one_pass, var_two_pass, rtol=1e-12)


def test_width_one_row_gives_beta():
    x = np.array([[3.0], [-2.0], [0.5]])
    y, mean, rstd = oracle.layernorm_fwd(x, np.array([2.0]), np.array([0.25]), EPS)
    np.testing.assert_array_equal(y, np.full((3, 1), 0.25))
    np.testing.assert_array_equal(mean, x[:, 0])


def test_bwd_matches_torch_autograd(ln_case):
    x, g, b, dy = ln_case
    dx, dg, db = oracle.layernorm_bwd(dy, x, g, EPS)
    xt = torch.from_numpy(x).requires_grad_()
    gt = torch.from_numpy(g).requires_grad_()
    bt = torch.from_numpy(b).requires_grad_()
    yt = torch.nn.functional.layer_norm(xt, (x.shape[1],), gt, bt, EPS)
    yt.backward(torch.from_numpy(dy))
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(db, bt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_bwd_matches_finite_differences():
    rng = np.random.default_rng(3)
    rows, cols = 3, 16
    x = rng.standard_normal((rows, cols))
    g = rng.normal(1.0, 0.1, cols)
    b = rng.normal(0.0, 0.1, cols)
    w = rng.standard_normal((rows, cols))
    dx, dg, db = oracle.layernorm_bwd(w, x, g, EPS)

    def loss(x_, g_, b_):
        return float((w * oracle.layernorm_fwd(x_, g_, b_, EPS)[0]).sum())

    h = 1e-6
    for arr, grad in [(x, dx), (g, dg), (b, db)]:
        num = np.zeros_like(arr)
        for k in np.ndindex(arr.shape):
            old = arr[k]
            arr[k] = old + h
            fp = loss(x, g, b)
            arr[k] = old - h
            fm = loss(x, g, b)
            arr[k] = old
            num[k] = (fp - fm) / (2 * h)
        assert np.abs(num - grad).max() <= 1e-6 * max(1.0, np.abs(grad).max())


def test_bwd_row_invariants(ln_case):
    # y does not change when x is shifted or scaled per row, so the gradient is
    # orthogonal to the all-ones vector and to xhat in every row.
    x, g, b, dy = ln_case
    dx, _, _ = oracle.layernorm_bwd(dy, x, g, EPS)
    _, mean, rstd = oracle.layernorm_fwd(x, g, b, 0.0)
    xhat = (x - mean[:, None]) * rstd[:, None]
    assert np.abs(dx.sum(axis=1)).max() <= 1e-12 * np.abs(dx).sum(axis=1).max()
    # With eps > 0 the scale invariance is broken by eps/(var+eps) only.
    _, _, rstd_eps = oracle.layernorm_fwd(x, g, b, EPS)
    var = 1.0 / rstd**2
    bound = 10 * EPS / var.min() * np.abs(dx * xhat).sum(axis=1).max()
    assert np.abs((dx * xhat).sum(axis=1)).max() <= bound + 1e-12


def test_bwd_equals_two_sum_form_of_the_pages(ln_case):
    # Slide p.22: dx from A = sum_j w_j dy_j and B = sum_j w_j dy_j x_j, computed
    # together, plus elementwise work:
    #   dx = rstd * (g - A/H - xhat * rstd * (B - mu*A)/H),  g = w * dy.
    x, gamma, b, dy = ln_case
    H = x.shape[1]
    dx, _, _ = oracle.layernorm_bwd(dy, x, gamma, EPS)
    _, mu, rstd = oracle.layernorm_fwd(x, gamma, b, EPS)
    gg = gamma[None, :] * dy
    A = gg.sum(axis=1, keepdims=True)
    B = (gg * x).sum(axis=1, keepdims=True)
    xhat = (x - mu[:, None]) * rstd[:, None]
    two_sum = rstd[:, None] * (gg - A / H - xhat * rstd[:, None] * (B - mu[:, None] * A) / H)
    np.testing.assert_allclose(dx, two_sum, rtol=1e-10, atol=1e-12)
