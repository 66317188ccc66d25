"""Pins for the oracle's masked attention softmax forward and backward.

Row softmax of the attention scores ("CS336 Lecture 5: GPU", section 6.1) with
the maximum subtracted (section 6.2), over the keys a padding mask and an
optional causal mask leave valid; "CMU 11-868 L10 (LightSeq)", slides p.23-26.
The oracle is pinned to torch in float64, to the online-softmax recurrence of
section 6.2, to finite differences and to closed forms.
"""
import numpy as np
import pytest
import torch

import oracle


def _valid(b, h, lq, lk, key_len, causal):
    v = np.ones((b, h, lq, lk), dtype=bool)
    j = np.arange(lk)
    if key_len is not None:
        kl = np.clip(np.asarray(key_len), 0, None)
        v &= (j[None, :] < kl[:, None])[:, None, None, :]
    if causal:
        q = np.arange(lq)
        v &= (j[None, :] <= (q[:, None] + lk - lq))[None, None, :, :]
    return v


CASES = [
    # (batch, heads, q_len, k_len, key_len, causal)
    (2, 3, 5, 16, [16, 9], False),
    (2, 2, 8, 8, None, True),
    (3, 1, 4, 12, [12, 0, 5], True),     # a fully masked batch element; q_len < k_len causal
    (1, 2, 6, 4, [3], True),             # q_len > k_len: early queries see no key
    (2, 1, 3, 1, [1, 1], False),         # one key per row
]


@pytest.mark.parametrize("case", CASES)
def test_fwd_matches_torch_masked_softmax(case):
    b, h, lq, lk, kl, causal = case
    x = np.random.default_rng(0).normal(0, 3, (b, h, lq, lk))
    y = oracle.softmax_fwd(x, kl, causal)
    valid = _valid(b, h, lq, lk, kl, causal)
    xt = torch.from_numpy(x).masked_fill(~torch.from_numpy(valid), float("-inf"))
    ref = torch.softmax(xt, dim=-1).nan_to_num(0.0).numpy()   # all-masked rows -> 0
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-15)
    assert (y[~valid] == 0.0).all()                            # exactly zero
    rows_with_key = valid.any(axis=-1)
    np.testing.assert_allclose(y.sum(axis=-1)[rows_with_key], 1.0, rtol=0, atol=1e-12)
    assert (y.sum(axis=-1)[~rows_with_key] == 0.0).all()


def test_shift_invariance_and_single_key():
    rng = np.random.default_rng(1)
    x = rng.normal(0, 3, (2, 2, 3, 10))
    y = oracle.softmax_fwd(x, [10, 4], False)
    y2 = oracle.softmax_fwd(x + rng.normal(0, 50, (2, 2, 3, 1)), [10, 4], False)
    np.testing.assert_allclose(y, y2, rtol=1e-10, atol=1e-14)
    one = oracle.softmax_fwd(rng.normal(0, 3, (1, 1, 4, 1)))
    np.testing.assert_array_equal(one, np.ones((1, 1, 4, 1)))


def test_causal_alignment_is_bottom_right():
    x = np.zeros((1, 1, 3, 5))
    y = oracle.softmax_fwd(x, None, True)
    # query q sees keys j <= q + (k_len - q_len) = q + 2
    want = np.array([[1 / 3] * 3 + [0, 0], [1 / 4] * 4 + [0], [1 / 5] * 5])
    np.testing.assert_allclose(y[0, 0], want, rtol=1e-15)


def test_fwd_equals_online_softmax_recurrence():
    # Section 6.2: running max m and normaliser l over tiles,
    #   m_t = max(m_{t-1}, max x^(t)),  l_t = l_{t-1} exp(m_{t-1} - m_t) + sum exp(x^(t) - m_t).
    rng = np.random.default_rng(2)
    lk, tile = 37, 8
    x = rng.normal(0, 3, (1, 1, 4, lk))
    y = oracle.softmax_fwd(x)
    for q in range(4):
        row = x[0, 0, q]
        m, l = -np.inf, 0.0
        for t0 in range(0, lk, tile):
            blk = row[t0:t0 + tile]
            m_new = max(m, blk.max())
            l = l * np.exp(m - m_new) + np.exp(blk - m_new).sum()
            m = m_new
        np.testing.assert_allclose(y[0, 0, q], np.exp(row - m) / l, rtol=1e-13)


@pytest.mark.parametrize("case", CASES)
def test_bwd_matches_torch_autograd(case):
    b, h, lq, lk, kl, causal = case
    rng = np.random.default_rng(4)
    x = rng.normal(0, 3, (b, h, lq, lk))
    dy = rng.standard_normal((b, h, lq, lk))
    y = oracle.softmax_fwd(x, kl, causal)
    dx = oracle.softmax_bwd(y, dy, kl, causal)
    valid = _valid(b, h, lq, lk, kl, causal)
    rows_with_key = valid.any(axis=-1, keepdims=True)
    # torch reference: softmax over valid entries only; rows without a key give 0.
    xt = torch.from_numpy(np.where(valid, x, 0.0)).requires_grad_()
    m = torch.from_numpy(valid)
    yt = torch.softmax(xt.masked_fill(~m, float("-inf")), -1).nan_to_num(0.0)
    yt = yt * torch.from_numpy(rows_with_key)
    yt.backward(torch.from_numpy(dy))
    ref = xt.grad.numpy() * valid
    np.testing.assert_allclose(dx, ref, rtol=1e-11, atol=1e-13)
    assert (dx[~valid] == 0.0).all()
    np.testing.assert_allclose(dx.sum(axis=-1), 0.0, atol=1e-12)


def test_bwd_matches_finite_differences():
    rng = np.random.default_rng(5)
    x = rng.normal(0, 3, (1, 2, 3, 7))
    w = rng.standard_normal(x.shape)
    kl = [5]
    y = oracle.softmax_fwd(x, kl, True)
    dx = oracle.softmax_bwd(y, w, kl, True)
    h = 1e-6
    num = np.zeros_like(x)
    for k in np.ndindex(x.shape):
        old = x[k]
        x[k] = old + h
        fp = float((w * oracle.softmax_fwd(x, kl, True)).sum())
        x[k] = old - h
        fm = float((w * oracle.softmax_fwd(x, kl, True)).sum())
        x[k] = old
        num[k] = (fp - fm) / (2 * h)
    assert np.abs(num - dx).max() <= 1e-6 * max(1.0, np.abs(dx).max())
