"""Pins of the oracle's embedding layer against numpy and the mathematics:
- at p = 0 the forward is numpy's gather s*E[tokens] + P[positions];
- its keep bits are the plain dropout bits over the output's flat index and
  kept values carry the 1/(1-p) scale;
- the backward equals numpy's unbuffered scatter-add (np.add.at) of the
  masked, scaled gradients, accumulates into an existing dE, and matches
  central finite differences of sum(w * y) in E."""
import numpy as np

import oracle

B, L, H, V, S = 2, 5, 16, 11, 2.5


def _case(seed):
    rng = np.random.default_rng(seed)
    tok = rng.integers(0, V, (B, L)).astype(np.int32)
    tok[0, :3] = 4  # a repeated token
    E = rng.normal(size=(V, H))
    P = rng.normal(size=(L + 3, H))
    return tok, E, P


def test_forward_is_a_gather_and_dropout():
    tok, E, P = _case(1)
    y0, w0 = oracle.embedding_fwd(tok, E, P, B, L, S, 0.0, 3, 4)
    ref = S * E[tok.ravel()] + P[np.tile(np.arange(L), B)]
    np.testing.assert_allclose(y0, ref, rtol=1e-15)
    assert (np.unpackbits(w0.view(np.uint8), bitorder="little")[: y0.size] == 1).all()
    y, w = oracle.embedding_fwd(tok, E, P, B, L, S, 0.25, 3, 4)
    np.testing.assert_array_equal(w, oracle.dropout_keep_bits(y.size, 0.25, 3, 4))
    bits = np.unpackbits(w.view(np.uint8), bitorder="little")[: y.size].astype(bool)
    np.testing.assert_allclose(y.ravel(), np.where(bits, ref.ravel() / (1 - np.float32(0.25)), 0),
                               rtol=1e-7)


def test_backward_is_a_scatter_add_and_accumulates():
    tok, E, P = _case(2)
    p = 0.25
    y, w = oracle.embedding_fwd(tok, E, P, B, L, S, p, 3, 4)
    dy = np.random.default_rng(5).normal(size=y.shape)
    bits = np.unpackbits(w.view(np.uint8), bitorder="little")[: y.size].reshape(y.shape)
    contrib = S * bits * dy / (1 - float(np.float32(p)))
    ref = np.zeros((V, H))
    np.add.at(ref, tok.ravel(), contrib)
    np.testing.assert_allclose(oracle.embedding_bwd(tok, dy, w, V, S, p), ref, rtol=1e-13,
                               atol=1e-15)
    base = np.random.default_rng(6).normal(size=(V, H))
    np.testing.assert_allclose(oracle.embedding_bwd(tok, dy, w, V, S, p, dE=base), base + ref,
                               rtol=1e-13, atol=1e-15)


def test_backward_finite_differences():
    tok, E, P = _case(3)
    p = 0.2
    _, w = oracle.embedding_fwd(tok, E, P, B, L, S, p, 7, 8)
    wt = np.random.default_rng(9).normal(size=(B * L, H))
    dE = oracle.embedding_bwd(tok, wt, w, V, S, p)
    h = 1e-6
    for (r, c) in [(4, 0), (4, 7), (int(tok[1, 2]), 3), (0, 15)]:
        Ep, Em = E.copy(), E.copy()
        Ep[r, c] += h
        Em[r, c] -= h
        fp = (wt * oracle.embedding_fwd(tok, Ep, P, B, L, S, p, 7, 8)[0]).sum()
        fm = (wt * oracle.embedding_fwd(tok, Em, P, B, L, S, p, 7, 8)[0]).sum()
        assert abs((fp - fm) / (2 * h) - dE[r, c]) < 1e-6
