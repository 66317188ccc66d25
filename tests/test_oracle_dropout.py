"""Pins for the oracle's bias+dropout+residual and bias+ReLU+dropout.

Fused operators from "CMU 11-868 L10 (LightSeq)", technique 1 (slide p.12),
and "LightSeq2 ..." section 2.1.1; the dropout mask m saved in the forward pass
and reused in the backward pass follows LightSeq2 section 2.1.2.
"""
import numpy as np
import pytest

import oracle


def _bits(words, n):
    return np.unpackbits(np.asarray(words, np.uint32).view(np.uint8), bitorder="little")[:n]


def _keep_by_word(n, p, seed, offset):
    thr = oracle.dropout_threshold(p)
    return np.array([oracle.dropout_word(seed, offset, i) >= thr for i in range(n)])


@pytest.fixture
def small():
    rng = np.random.default_rng(0)
    rows, cols = 6, 20  # 120 elements: 3 full mask words and a ragged 24-bit tail
    x = rng.standard_normal((rows, cols))
    bias = rng.normal(0, 0.02, cols)
    res = rng.standard_normal((rows, cols))
    return x, bias, res


def test_bdr_p0_is_plain_sum(small):
    x, bias, res = small
    out, mask = oracle.bias_dropout_residual_fwd(x, bias, res, 0.0, 0, 0)
    np.testing.assert_allclose(out, res + x + bias[None, :], rtol=0, atol=1e-15)
    assert _bits(mask, x.size).all()
    assert (mask[-1] >> (x.size % 32)) == 0  # bits past the last element are 0


def test_bdr_each_element_dropped_or_scaled(small):
    x, bias, res = small
    p, seed, off = 0.3, 7, 2
    out, mask = oracle.bias_dropout_residual_fwd(x, bias, res, p, seed, off)
    keep = _keep_by_word(x.size, p, seed, off).reshape(x.shape)
    np.testing.assert_array_equal(_bits(mask, x.size).reshape(x.shape).astype(bool), keep)
    want = np.where(keep, res + (x + bias[None, :]) / (1.0 - np.float64(np.float32(p))), res)
    np.testing.assert_allclose(out, want, rtol=1e-15, atol=1e-15)
    assert 0 < keep.sum() < keep.size


def _fd_check(f, args, idx, grad, h=1e-6, rtol=1e-6):
    """Central differences of scalar f with respect to args[idx], against grad."""
    a = [np.array(v, dtype=np.float64, copy=True) for v in args]
    num = np.zeros_like(a[idx])
    it = np.nditer(a[idx], flags=["multi_index"])
    for _ in it:
        k = it.multi_index
        old = a[idx][k]
        a[idx][k] = old + h
        fp = f(*a)
        a[idx][k] = old - h
        fm = f(*a)
        a[idx][k] = old
        num[k] = (fp - fm) / (2 * h)
    scale = max(1.0, np.abs(grad).max())
    assert np.abs(num - grad).max() <= rtol * scale + 1e-9, np.abs(num - grad).max()


def test_bdr_bwd_matches_finite_differences(small):
    x, bias, res = small
    p, seed, off = 0.25, 1, 9
    w = np.random.default_rng(5).standard_normal(x.shape)  # L = <w, out>

    def loss(x_, b_, r_):
        out, _ = oracle.bias_dropout_residual_fwd(x_, b_, r_, p, seed, off)
        return float((w * out).sum())

    _, mask = oracle.bias_dropout_residual_fwd(x, bias, res, p, seed, off)
    dx, db = oracle.bias_dropout_residual_bwd(w, mask, p)
    _fd_check(loss, [x, bias, res], 0, dx)
    _fd_check(loss, [x, bias, res], 1, db)
    _fd_check(loss, [x, bias, res], 2, w)  # d residual = d out
    # Drawing the bits again from (seed, offset) gives the same gradient.
    dx2, db2 = oracle.bias_dropout_residual_bwd(w, None, p, seed, off)
    np.testing.assert_array_equal(dx, dx2)
    np.testing.assert_array_equal(db, db2)


def test_brd_p0_is_relu_and_mask_is_relu_pattern(small):
    x, bias, _ = small
    x = x.copy()
    x[0, 3] = -bias[3]  # z == 0 exactly: ReLU(0) = 0 and its bit is 0
    out, mask = oracle.bias_relu_dropout_fwd(x, bias, 0.0, 0, 0)
    z = x + bias[None, :]
    np.testing.assert_allclose(out, np.maximum(z, 0.0), rtol=0, atol=0)
    np.testing.assert_array_equal(_bits(mask, x.size).reshape(x.shape).astype(bool), z > 0)
    assert not _bits(mask, x.size)[3]


def test_brd_large_positive_input_gives_bdr_keep_pattern(small):
    x, bias, res = small
    p, seed, off = 0.4, 12, 3
    xp = np.abs(x) + 100.0
    _, m_brd = oracle.bias_relu_dropout_fwd(xp, bias, p, seed, off)
    _, m_bdr = oracle.bias_dropout_residual_fwd(xp, bias, res, p, seed, off)
    np.testing.assert_array_equal(m_brd, m_bdr)


def test_brd_bwd_matches_finite_differences(small):
    x, bias, _ = small
    x = x + np.sign(x) * 0.05  # keep z away from the ReLU kink for the difference quotient
    p, seed, off = 0.2, 4, 4
    w = np.random.default_rng(6).standard_normal(x.shape)

    def loss(x_, b_):
        out, _ = oracle.bias_relu_dropout_fwd(x_, b_, p, seed, off)
        return float((w * out).sum())

    _, mask = oracle.bias_relu_dropout_fwd(x, bias, p, seed, off)
    dx, db = oracle.bias_relu_dropout_bwd(w, mask, p)
    _fd_check(loss, [x, bias], 0, dx)
    _fd_check(loss, [x, bias], 1, db)


def test_bias_grad_is_column_sum_not_row_sum():
    # A transposed reduction (over columns instead of rows) would fail here.
    rows, cols = 3, 8
    dout = np.arange(rows * cols, dtype=np.float64).reshape(rows, cols)
    words = oracle.dropout_keep_bits(rows * cols, 0.0, 0, 0)
    dx, db = oracle.bias_dropout_residual_bwd(dout, words, 0.0)
    np.testing.assert_array_equal(dx, dout)
    np.testing.assert_array_equal(db, dout.sum(axis=0))
