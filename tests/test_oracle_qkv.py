"""Pins of the oracle's bias + reshape of Q, K, V against what the layout and
the mathematics fix:
- the forward equals numpy's own reshape [batch, seq, 3, heads, d] ->
  transpose to [3, batch, heads, seq, d], plus the bias broadcast;
- the backward is the adjoint of the bias-free forward (dot-product test) and
  undoes it exactly; dbias is the column sum of dqkv;
- a one-hot input lands at the single place its indices name."""
import numpy as np
import pytest

import oracle

SHAPES = [(2, 3, 4, 8), (1, 1, 1, 8), (3, 5, 2, 16)]


@pytest.mark.parametrize("shape", SHAPES)
def test_forward_is_numpy_reshape_plus_bias(shape):
    B, L, h, d = shape
    rng = np.random.default_rng(0)
    x = rng.normal(size=(B * L, 3 * h * d))
    b = rng.normal(size=3 * h * d)
    got = oracle.bias_reshape_qkv_fwd(x, b, B, L, h, d)
    ref = (x + b).reshape(B, L, 3, h, d).transpose(2, 0, 3, 1, 4)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("shape", SHAPES)
def test_backward_is_the_adjoint_and_inverse(shape):
    B, L, h, d = shape
    rng = np.random.default_rng(1)
    x = rng.normal(size=(B * L, 3 * h * d))
    y = rng.normal(size=(3, B, h, L, d))
    fx = oracle.bias_reshape_qkv_fwd(x, np.zeros(3 * h * d), B, L, h, d)
    gy, db = oracle.bias_reshape_qkv_bwd(y, B, L, h, d)
    assert np.isclose(np.vdot(fx, y), np.vdot(x, gy), rtol=1e-12)
    back, _ = oracle.bias_reshape_qkv_bwd(fx, B, L, h, d)
    np.testing.assert_array_equal(back, x)
    np.testing.assert_allclose(db, gy.sum(axis=0), rtol=1e-13)


def test_one_hot_lands_where_its_indices_say():
    B, L, h, d = 2, 3, 4, 8
    H = h * d
    for (b, l, s, hh, j) in [(0, 0, 0, 0, 0), (1, 2, 2, 3, 7), (1, 0, 1, 2, 5)]:
        x = np.zeros((B * L, 3 * H))
        x[b * L + l, s * H + hh * d + j] = 1.0
        out = oracle.bias_reshape_qkv_fwd(x, np.zeros(3 * H), B, L, h, d)
        assert out[s, b, hh, l, j] == 1.0 and out.sum() == 1.0
