"""Algorithmic HBM bytes of each fused operator, and roofline arithmetic.

A fused kernel's algorithmic traffic is every input read once plus every
output written once, at storage size ("CMU 11-868 L10 (LightSeq)", intuition
section, slide p.10: E = A + B + D as one kernel is 3 reads and 1 write, as two
kernels 4 reads and 2 writes; "CS336 Lecture 5: GPU", section 4.3: a fused
LayerNorm+GELU+dropout moves 2 x size(x) instead of 6 x).  Scratch traffic a
kernel adds on top (partial sums of column reductions) is not algorithmic and
is not counted.  Roofline: P = min(pi, beta * AI) with AI = FLOPs / bytes
("CS336 Lecture 5: GPU", sections 2.1-2.2).
"""
from __future__ import annotations

from typing import Dict, Iterable, Optional

import numpy as np

MASK_BYTES_PER_ELEM = 1.0 / 8.0  # one bit per element


def traffic(reads: Iterable[float], writes: Iterable[float]) -> float:
    """Bytes moved by a kernel that reads and writes the given buffer sizes once."""
    return float(sum(reads)) + float(sum(writes))


def unfused_chain_traffic(n_inputs: int, size: float) -> float:
    """An n-ary elementwise chain as n-1 binary kernels, each reading two
    operands and writing one result of `size` bytes."""
    kernels = n_inputs - 1
    return kernels * traffic([size, size], [size])


def arithmetic_intensity(flops: float, nbytes: float) -> float:
    return flops / nbytes


def ridge_point(peak_flops: float, bandwidth: float) -> float:
    return peak_flops / bandwidth


def attainable(peak_flops: float, bandwidth: float, ai: float) -> float:
    return min(peak_flops, bandwidth * ai)


# --- the operators -------------------------------------------------------
def bdr_fwd_bytes(rows: int, cols: int, esize: int, with_mask: bool = True) -> float:
    n = rows * cols
    return traffic([n * esize, n * esize, cols * esize],
                   [n * esize] + ([n * MASK_BYTES_PER_ELEM] if with_mask else []))


def dropout_bwd_bytes(rows: int, cols: int, esize: int, with_mask: bool = True,
                      with_dbias: bool = True) -> float:
    n = rows * cols
    return traffic([n * esize] + ([n * MASK_BYTES_PER_ELEM] if with_mask else []),
                   [n * esize] + ([cols * esize] if with_dbias else []))


def brd_fwd_bytes(rows: int, cols: int, esize: int) -> float:
    n = rows * cols
    return traffic([n * esize, cols * esize], [n * esize, n * MASK_BYTES_PER_ELEM])


def ln_fwd_bytes(rows: int, cols: int, esize: int) -> float:
    n = rows * cols
    return traffic([n * esize, 2 * cols * esize], [n * esize, 8 * rows])


def ln_bwd_bytes(rows: int, cols: int, esize: int) -> float:
    n = rows * cols
    return traffic([2 * n * esize, cols * esize, 8 * rows], [n * esize, 2 * cols * esize])


def softmax_valid_count(batch: int, heads: int, q_len: int, k_len: int,
                        key_len: Optional[np.ndarray], causal: bool) -> int:
    """Number of valid (unmasked) entries of a [batch, heads, q_len, k_len] score tensor."""
    q = np.arange(q_len)
    per_q = np.full(q_len, k_len, dtype=np.int64)
    if causal:
        per_q = np.clip(q + k_len - q_len + 1, 0, k_len)
    if key_len is None:
        return int(per_q.sum()) * batch * heads
    kl = np.clip(np.asarray(key_len, dtype=np.int64), 0, k_len)
    return int(np.minimum(per_q[None, :], kl[:, None]).sum()) * heads


def softmax_fwd_bytes(batch, heads, q_len, k_len, esize, key_len=None, causal=False) -> float:
    valid = softmax_valid_count(batch, heads, q_len, k_len, key_len, causal)
    rows = batch * heads * q_len
    return traffic([valid * esize] + ([4 * batch] if key_len is not None else []),
                   [rows * k_len * esize])


def softmax_bwd_bytes(batch, heads, q_len, k_len, esize, key_len=None, causal=False) -> float:
    valid = softmax_valid_count(batch, heads, q_len, k_len, key_len, causal)
    rows = batch * heads * q_len
    return traffic([2 * valid * esize] + ([4 * batch] if key_len is not None else []),
                   [rows * k_len * esize])


def softmax_dropout_fwd_bytes(batch, heads, q_len, k_len, esize, key_len=None,
                              causal=False) -> float:
    """Softmax with dropout on the probabilities: the valid scores in; y and
    y_drop (whole rows) and one mask bit per element out."""
    valid = softmax_valid_count(batch, heads, q_len, k_len, key_len, causal)
    n = batch * heads * q_len * k_len
    return traffic([valid * esize] + ([4 * batch] if key_len is not None else []),
                   [2 * n * esize, n * MASK_BYTES_PER_ELEM])


def softmax_dropout_bwd_bytes(batch, heads, q_len, k_len, esize, key_len=None,
                              causal=False) -> float:
    """Its backward: y, dy_drop and the mask bits of the valid entries in; dx out."""
    valid = softmax_valid_count(batch, heads, q_len, k_len, key_len, causal)
    n = batch * heads * q_len * k_len
    return traffic([2 * valid * esize, valid * MASK_BYTES_PER_ELEM] +
                   ([4 * batch] if key_len is not None else []), [n * esize])


def qkv_fwd_bytes(rows: int, cols: int, esize: int) -> float:
    """Bias + reshape of Q, K, V over [rows, cols = 3H]: each value read and written once."""
    n = rows * cols
    return traffic([n * esize, cols * esize], [n * esize])


def qkv_bwd_bytes(rows: int, cols: int, esize: int) -> float:
    n = rows * cols
    return traffic([n * esize], [n * esize, cols * esize])


def cross_entropy_fwd_bytes(rows: int, vocab: int, esize: int) -> float:
    """Logits and targets in; loss and lse (FP32) out."""
    return traffic([rows * vocab * esize, 4 * rows], [8 * rows])


def cross_entropy_bwd_bytes(rows: int, vocab: int, esize: int) -> float:
    """Logits, targets, lse and the upstream gradient in; logit gradients out."""
    return traffic([rows * vocab * esize, 12 * rows], [rows * vocab * esize])


def embedding_fwd_bytes(tokens: int, seq: int, hidden: int, esize: int) -> float:
    """Ids in; one token-table row per token and the position table once in;
    y and its mask bits out."""
    return traffic([4 * tokens, tokens * hidden * esize, seq * hidden * esize],
                   [tokens * hidden * esize, tokens * hidden * MASK_BYTES_PER_ELEM])


def embedding_bwd_bytes(tokens: int, unique: int, hidden: int, esize: int) -> float:
    """dy, its mask bits and the ids in; each touched FP32 table-gradient row
    read and written once."""
    return traffic([4 * tokens, tokens * hidden * esize, tokens * hidden * MASK_BYTES_PER_ELEM,
                    4 * unique * hidden], [4 * unique * hidden])


def adam_bytes(n: int, esize: int) -> float:
    """Trainer update: parameters and gradients in the storage dtype, FP32 moments."""
    return traffic([n * esize, n * esize, 4 * n, 4 * n], [n * esize, 4 * n, 4 * n])


def layer_step_bytes(tokens: int, hidden: int, ffn: int, batch: int, heads: int, seq: int,
                     esize: int, key_len=None, causal=False) -> Dict[str, float]:
    """Algorithmic bytes of every operator of one layer's forward and backward
    (two bias+dropout+residual, one bias+ReLU+dropout, two LayerNorms, one
    softmax, each forward and backward)."""
    T, H, F = tokens, hidden, ffn
    sm = dict(batch=batch, heads=heads, q_len=seq, k_len=seq, esize=esize, key_len=key_len,
              causal=causal)
    return {
        "softmax_fwd": softmax_fwd_bytes(**sm),
        "attn_bdr_fwd": bdr_fwd_bytes(T, H, esize),
        "ln1_fwd": ln_fwd_bytes(T, H, esize),
        "ffn1_brd_fwd": brd_fwd_bytes(T, F, esize),
        "ffn2_bdr_fwd": bdr_fwd_bytes(T, H, esize),
        "ln2_fwd": ln_fwd_bytes(T, H, esize),
        "ln2_bwd": ln_bwd_bytes(T, H, esize),
        "ffn2_bdr_bwd": dropout_bwd_bytes(T, H, esize),
        "ffn1_brd_bwd": dropout_bwd_bytes(T, F, esize),
        "ln1_bwd": ln_bwd_bytes(T, H, esize),
        "attn_bdr_bwd": dropout_bwd_bytes(T, H, esize),
        "softmax_bwd": softmax_bwd_bytes(**sm),
    }


def layer_step_read_write(tokens: int, hidden: int, ffn: int, batch: int, heads: int, seq: int,
                          esize: int, key_len=None, causal=False) -> Dict[str, tuple]:
    """(read bytes, write bytes) of every operator of layer_step_bytes, for a
    plain streaming copy that moves the same bytes (the floor a dependent
    launch of that size can reach)."""
    T, H, F = tokens, hidden, ffn
    n_h, n_f = T * H, T * F
    m = MASK_BYTES_PER_ELEM
    sm = dict(batch=batch, heads=heads, q_len=seq, k_len=seq, key_len=key_len, causal=causal)
    valid = softmax_valid_count(**sm)
    dense = batch * heads * seq * seq
    kl = 4 * batch if key_len is not None else 0
    rw = {
        "softmax_fwd": (valid * esize + kl, dense * esize),
        "attn_bdr_fwd": (2 * n_h * esize + H * esize, n_h * esize + n_h * m),
        "ln1_fwd": (n_h * esize + 2 * H * esize, n_h * esize + 8 * T),
        "ffn1_brd_fwd": (n_f * esize + F * esize, n_f * esize + n_f * m),
        "ffn2_bdr_fwd": (2 * n_h * esize + H * esize, n_h * esize + n_h * m),
        "ln2_fwd": (n_h * esize + 2 * H * esize, n_h * esize + 8 * T),
        "ln2_bwd": (2 * n_h * esize + H * esize + 8 * T, n_h * esize + 2 * H * esize),
        "ffn2_bdr_bwd": (n_h * esize + n_h * m, n_h * esize + H * esize),
        "ffn1_brd_bwd": (n_f * esize + n_f * m, n_f * esize + F * esize),
        "ln1_bwd": (2 * n_h * esize + H * esize + 8 * T, n_h * esize + 2 * H * esize),
        "attn_bdr_bwd": (n_h * esize + n_h * m, n_h * esize + H * esize),
        "softmax_bwd": (2 * valid * esize + kl, dense * esize),
    }
    return {k: (float(r), float(w)) for k, (r, w) in rw.items()}
