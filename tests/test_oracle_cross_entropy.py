"""Pins of the oracle's cross entropy against an independent library and the
mathematics:
- torch.nn.functional.cross_entropy in float64 (reduction 'none'), with and
  without label smoothing and an ignore index, and its autograd gradient;
- central finite differences of the loss;
- each gradient row sums to 0 (softmax minus a distribution summing to 1);
- uniform logits give loss log V and constant shifts change nothing."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
F = torch.nn.functional


def _case(seed, rows=7, V=40):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 3, (rows, V))
    t = rng.integers(0, V, rows).astype(np.int32)
    return z, t


@pytest.mark.parametrize("eps", [0.0, 0.1])
def test_matches_torch_cross_entropy(eps):
    z, t = _case(1)
    t[2] = -100  # ignored
    loss, lse = oracle.cross_entropy_fwd(z, t, eps, -100)
    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    ref = F.cross_entropy(zt, torch.tensor(t, dtype=torch.int64), reduction="none",
                          label_smoothing=eps, ignore_index=-100)
    np.testing.assert_allclose(loss, ref.detach().numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, torch.logsumexp(zt, 1).detach().numpy(), rtol=1e-13)
    g = np.random.default_rng(2).normal(size=len(t))
    ref.backward(torch.tensor(g))
    dz = oracle.cross_entropy_bwd(z, t, g, eps, -100)
    np.testing.assert_allclose(dz, zt.grad.numpy(), rtol=1e-11, atol=1e-14)


def test_finite_differences_and_row_sums():
    z, t = _case(3, rows=3, V=12)
    eps = 0.2
    dz = oracle.cross_entropy_bwd(z, t, None, eps)
    h = 1e-6
    for idx in np.ndindex(z.shape):
        zp, zm = z.copy(), z.copy()
        zp[idx] += h
        zm[idx] -= h
        num = (oracle.cross_entropy_fwd(zp, t, eps)[0].sum()
               - oracle.cross_entropy_fwd(zm, t, eps)[0].sum()) / (2 * h)
        assert abs(num - dz[idx]) < 1e-7
    np.testing.assert_allclose(dz.sum(axis=1), 0.0, atol=1e-14)


def test_uniform_logits_and_shift_invariance():
    V = 64
    z = np.zeros((2, V))
    t = np.array([3, 60], dtype=np.int32)
    loss, lse = oracle.cross_entropy_fwd(z, t, 0.0)
    np.testing.assert_allclose(loss, np.log(V), rtol=1e-15)
    z2, t2 = _case(4)
    a = oracle.cross_entropy_fwd(z2, t2, 0.1)[0]
    b = oracle.cross_entropy_fwd(z2 + 1234.5, t2, 0.1)[0]
    np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-11)


def test_out_of_range_targets_are_ignored():
    z, t = _case(5)
    t[0], t[1] = -1, 40
    loss, _ = oracle.cross_entropy_fwd(z, t, 0.0, -100)
    assert loss[0] == 0.0 and loss[1] == 0.0
    dz = oracle.cross_entropy_bwd(z, t, None, 0.0, -100)
    assert not dz[:2].any()
