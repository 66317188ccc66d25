"""Pins of the oracle's softmax with fused dropout on the probabilities:
- its y is the plain softmax, and with p = 0 y_drop is y and the bits are
  exactly the valid entries (y > 0; masked entries are exact zeros);
- its bits are the plain dropout keep bits (the pinned Philox stream over the
  flat index) restricted to the valid entries, kept at a rate within 3 sigma
  of 1 - p;
- the backward matches central finite differences of sum(w * y_drop(x)) with
  the bits fixed, reduces to the plain softmax backward at p = 0, and its
  rows sum to 0."""
import numpy as np
import pytest

import oracle

P, SEED, OFF = 0.3, 17, 5


def _case(seed, b=2, h=3, lq=5, lk=16, causal=False, pad=True):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 3, (b, h, lq, lk))
    kl = rng.integers(1, lk + 1, b).astype(np.int32) if pad else None
    return x, kl, causal


@pytest.mark.parametrize("causal,pad", [(False, True), (True, False), (True, True)])
def test_forward_composition_and_p_zero(causal, pad):
    x, kl, c = _case(1, causal=causal, pad=pad)
    y, yd, w = oracle.softmax_dropout_fwd(x, kl, c, P, SEED, OFF)
    np.testing.assert_array_equal(y, oracle.softmax_fwd(x, kl, c))
    keep = oracle.dropout_keep_bits(x.size, P, SEED, OFF)
    bits = np.unpackbits(w.view(np.uint8), bitorder="little")[: x.size].astype(bool)
    kbits = np.unpackbits(keep.view(np.uint8), bitorder="little")[: x.size].astype(bool)
    valid = (y > 0).ravel()
    np.testing.assert_array_equal(bits, kbits & valid)
    scale = 1.0 / (1.0 - float(np.float32(P)))  # p is passed as FP32, scaled in FP64
    np.testing.assert_array_equal(yd.ravel(), np.where(bits, y.ravel() * scale, 0.0))
    y0, yd0, w0 = oracle.softmax_dropout_fwd(x, kl, c, 0.0, SEED, OFF)
    np.testing.assert_array_equal(yd0, y0)
    np.testing.assert_array_equal(np.unpackbits(w0.view(np.uint8), bitorder="little")[: x.size]
                                  .astype(bool), valid)


def test_keep_rate_on_valid_entries():
    x, kl, c = _case(2, b=8, h=8, lq=16, lk=64)
    y, _, w = oracle.softmax_dropout_fwd(x, kl, c, P, SEED, OFF)
    bits = np.unpackbits(w.view(np.uint8), bitorder="little")[: x.size].astype(bool)
    valid = (y > 0).ravel()
    n = valid.sum()
    rate = bits[valid].mean()
    assert abs(rate - (1 - P)) <= 3 * np.sqrt(P * (1 - P) / n)
    assert not bits[~valid].any()


@pytest.mark.parametrize("causal,pad", [(False, True), (True, True)])
def test_backward_finite_differences(causal, pad):
    x, kl, c = _case(3, b=1, h=2, lq=3, lk=8, causal=causal, pad=pad)
    y, _, w = oracle.softmax_dropout_fwd(x, kl, c, P, SEED, OFF)
    wt = np.random.default_rng(4).normal(size=x.shape)
    dx = oracle.softmax_dropout_bwd(y, wt, w, kl, c, P)
    h = 1e-6
    num = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        # the bits stay fixed: the same (seed, offset) and the same valid set
        fp = (wt * oracle.softmax_dropout_fwd(xp, kl, c, P, SEED, OFF)[1]).sum()
        fm = (wt * oracle.softmax_dropout_fwd(xm, kl, c, P, SEED, OFF)[1]).sum()
        num[idx] = (fp - fm) / (2 * h)
    np.testing.assert_allclose(dx, num, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dx.sum(axis=-1), 0.0, atol=1e-12)


def test_backward_at_p_zero_is_the_softmax_backward():
    x, kl, c = _case(5)
    y, _, w = oracle.softmax_dropout_fwd(x, kl, c, 0.0, SEED, OFF)
    dy = np.random.default_rng(6).normal(size=x.shape)
    np.testing.assert_allclose(oracle.softmax_dropout_bwd(y, dy, w, kl, c, 0.0),
                               oracle.softmax_bwd(y, dy, kl, c), rtol=1e-14, atol=1e-16)
