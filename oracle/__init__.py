"""FP64 CPU oracle for the fused non-GEMM Transformer-layer operators.

TEST INFRASTRUCTURE ONLY.  The plain C definitions in ``ls_oracle.c`` are what
the CUDA library is checked against.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package; the product path never does.  Nothing here imports the CUDA library
or shares code with it.

Every function takes numpy arrays holding exactly the values the GPU gets
(FP16/FP32 storage values, widened to float64) and returns float64 results.
Dropout masks are ``uint32`` word arrays: element ``i`` is bit ``i & 31`` of
word ``i >> 5``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libls_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ls_oracle.c`` with gcc into ``oracle/_build/libls_oracle.so``."""
    src = os.path.join(_HERE, "ls_oracle.c")
    hdr = os.path.join(_HERE, "ls_oracle.h")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(src), os.path.getmtime(hdr))):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -O2 without -ffast-math: the arithmetic stays IEEE double, in source order.
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
           "-fPIC", "-shared", "-Wall", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i64, f32, f64, u64, u32, cint = (ctypes.c_int64, ctypes.c_float, ctypes.c_double,
                                      ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int)
    sig = {
        "or_philox4x32_10": (None, [P, P, P]),
        "or_dropout_word": (u32, [u64, u64, u64]),
        "or_dropout_threshold": (u32, [f32]),
        "or_dropout_keep_bits": (None, [i64, f32, u64, u64, P]),
        "or_bdr_fwd": (None, [i64, i64, P, P, P, f32, u64, u64, P, P]),
        "or_bdr_bwd": (None, [i64, i64, P, P, f32, u64, u64, P, P]),
        "or_brd_fwd": (None, [i64, i64, P, P, f32, u64, u64, P, P]),
        "or_brd_bwd": (None, [i64, i64, P, P, f32, P, P]),
        "or_layernorm_fwd": (None, [i64, i64, P, P, P, f64, P, P, P]),
        "or_layernorm_bwd": (None, [i64, i64, P, P, P, f64, P, P, P]),
        "or_softmax_fwd": (None, [i64, i64, i64, i64, P, P, cint, P]),
        "or_softmax_bwd": (None, [i64, i64, i64, i64, P, P, P, cint, P]),
        "or_num_threads": (cint, []),
        "or_set_num_threads": (None, [cint]),
        "or_adam_update": (None, [i64, P, P, P, P, f64, f64, f64, f64, f64, i64, f64, P, P, P]),
        "or_bias_reshape_qkv_fwd": (None, [i64, i64, i64, i64, P, P, P]),
        "or_embedding_fwd": (None, [i64, i64, i64, i64, P, P, P, f64, f32, u64, u64, P, P]),
        "or_embedding_bwd": (None, [i64, i64, i64, P, P, P, f64, f32, P]),
        "or_cross_entropy_fwd": (None, [i64, i64, P, P, f64, ctypes.c_int32, P, P]),
        "or_cross_entropy_bwd": (None, [i64, i64, P, P, P, f64, ctypes.c_int32, P]),
        "or_softmax_dropout_fwd": (None, [i64, i64, i64, i64, P, P, cint, f32, u64, u64, P, P, P]),
        "or_softmax_dropout_bwd": (None, [i64, i64, i64, i64, P, P, P, P, cint, f32, P]),
        "or_bias_reshape_qkv_bwd": (None, [i64, i64, i64, i64, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def mask_words(n: int) -> int:
    """Number of uint32 words a mask of n elements occupies."""
    return (n + 31) // 32


def num_threads() -> int:
    return _load().or_num_threads()


def set_num_threads(n: int) -> None:
    """Threads for the row loops of later calls (OpenMP)."""
    _load().or_set_num_threads(int(n))


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    _load().or_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def dropout_word(seed: int, offset: int, i: int) -> int:
    return int(_load().or_dropout_word(seed, offset, i))


def dropout_threshold(p: float) -> int:
    return int(_load().or_dropout_threshold(p))


def dropout_keep_bits(n: int, p: float, seed: int, offset: int) -> np.ndarray:
    w = np.zeros(mask_words(n), dtype=np.uint32)
    _load().or_dropout_keep_bits(n, p, seed, offset, _ptr(w))
    return w


def bias_dropout_residual_fwd(x, bias, residual, p, seed, offset):
    """Returns (out, mask_words) for out = residual + keep * (x + bias) / (1 - p)."""
    x, bias, residual = _f64(x), _f64(bias), _f64(residual)
    rows, cols = x.shape
    out = np.empty_like(x)
    mask = np.zeros(mask_words(rows * cols), dtype=np.uint32)
    _load().or_bdr_fwd(rows, cols, _ptr(x), _ptr(bias), _ptr(residual), p, seed, offset,
                       _ptr(out), _ptr(mask))
    return out, mask


def bias_dropout_residual_bwd(dout, mask, p, seed=0, offset=0):
    """Returns (dx, dbias).  mask=None draws the keep bits again from (seed, offset)."""
    dout = _f64(dout)
    rows, cols = dout.shape
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint32)
    dx = np.empty_like(dout)
    db = np.empty(cols, dtype=np.float64)
    _load().or_bdr_bwd(rows, cols, _ptr(dout), _ptr(m), p, seed, offset, _ptr(dx), _ptr(db))
    return dx, db


def bias_relu_dropout_fwd(x, bias, p, seed, offset):
    """Returns (out, mask_words) for out = ((z > 0) and keep) * z / (1 - p), z = x + bias."""
    x, bias = _f64(x), _f64(bias)
    rows, cols = x.shape
    out = np.empty_like(x)
    mask = np.zeros(mask_words(rows * cols), dtype=np.uint32)
    _load().or_brd_fwd(rows, cols, _ptr(x), _ptr(bias), p, seed, offset, _ptr(out), _ptr(mask))
    return out, mask


def bias_relu_dropout_bwd(dout, mask, p):
    dout = _f64(dout)
    rows, cols = dout.shape
    m = np.ascontiguousarray(mask, dtype=np.uint32)
    dx = np.empty_like(dout)
    db = np.empty(cols, dtype=np.float64)
    _load().or_brd_bwd(rows, cols, _ptr(dout), _ptr(m), p, _ptr(dx), _ptr(db))
    return dx, db


def layernorm_fwd(x, gamma, beta, eps):
    """Returns (y, mean, rstd)."""
    x, gamma, beta = _f64(x), _f64(gamma), _f64(beta)
    rows, cols = x.shape
    y = np.empty_like(x)
    mean = np.empty(rows)
    rstd = np.empty(rows)
    _load().or_layernorm_fwd(rows, cols, _ptr(x), _ptr(gamma), _ptr(beta), float(eps),
                             _ptr(y), _ptr(mean), _ptr(rstd))
    return y, mean, rstd


def layernorm_bwd(dy, x, gamma, eps):
    """Returns (dx, dgamma, dbeta); the row statistics are recomputed from x."""
    dy, x, gamma = _f64(dy), _f64(x), _f64(gamma)
    rows, cols = x.shape
    dx = np.empty_like(x)
    dg = np.empty(cols)
    db = np.empty(cols)
    _load().or_layernorm_bwd(rows, cols, _ptr(dy), _ptr(x), _ptr(gamma), float(eps),
                             _ptr(dx), _ptr(dg), _ptr(db))
    return dx, dg, db


def _key_len(key_len):
    if key_len is None:
        return None
    return np.ascontiguousarray(np.asarray(key_len, dtype=np.int32))


def softmax_fwd(x, key_len=None, causal=False):
    """x: [batch, heads, q_len, k_len].  Returns y of the same shape."""
    x = _f64(x)
    b, h, lq, lk = x.shape
    kl = _key_len(key_len)
    y = np.empty_like(x)
    _load().or_softmax_fwd(b, h, lq, lk, _ptr(x), _ptr(kl), int(bool(causal)), _ptr(y))
    return y


def softmax_bwd(y, dy, key_len=None, causal=False):
    y, dy = _f64(y), _f64(dy)
    b, h, lq, lk = y.shape
    kl = _key_len(key_len)
    dx = np.empty_like(y)
    _load().or_softmax_bwd(b, h, lq, lk, _ptr(y), _ptr(dy), _ptr(kl), int(bool(causal)), _ptr(dx))
    return dx


def adam_update(p, g, m, v, lr, beta1, beta2, eps, weight_decay, step, grad_scale=1.0):
    """One trainer update of a flat workspace: returns (p', m', v') in float64.
    Hyperparameters are taken as given (pass the FP32 values the GPU gets)."""
    p, g, m, v = (_f64(a).ravel() for a in (p, g, m, v))
    n = p.size
    assert g.size == n and m.size == n and v.size == n
    po, mo, vo = np.empty(n), np.empty(n), np.empty(n)
    _load().or_adam_update(n, _ptr(p), _ptr(g), _ptr(m), _ptr(v), float(lr), float(beta1),
                           float(beta2), float(eps), float(weight_decay), int(step),
                           float(grad_scale), _ptr(po), _ptr(mo), _ptr(vo))
    return po, mo, vo


def bias_reshape_qkv_fwd(qkv, bias, batch, seq, heads, d):
    """qkv [batch*seq, 3*heads*d] + bias -> [3, batch, heads, seq, d] (float64)."""
    x, b = _f64(qkv), _f64(bias)
    assert x.size == batch * seq * 3 * heads * d and b.size == 3 * heads * d
    out = np.empty((3, batch, heads, seq, d))
    _load().or_bias_reshape_qkv_fwd(batch, seq, heads, d, _ptr(x), _ptr(b), _ptr(out))
    return out


def bias_reshape_qkv_bwd(dout, batch, seq, heads, d):
    """dout [3, batch, heads, seq, d] -> (dqkv [batch*seq, 3*heads*d], dbias [3*heads*d])."""
    g = _f64(dout)
    assert g.size == 3 * batch * heads * seq * d
    dqkv = np.empty((batch * seq, 3 * heads * d))
    dbias = np.empty(3 * heads * d)
    _load().or_bias_reshape_qkv_bwd(batch, seq, heads, d, _ptr(g), _ptr(dqkv), _ptr(dbias))
    return dqkv, dbias


def softmax_dropout_fwd(x, key_len, causal, p, seed, offset):
    """Returns (y, y_drop, mask_words) for scores x [batch, heads, q_len, k_len]."""
    xx = _f64(x)
    b, h, lq, lk = xx.shape
    kl = _key_len(key_len)
    y, yd = np.empty_like(xx), np.empty_like(xx)
    w = np.zeros(mask_words(xx.size), dtype=np.uint32)
    _load().or_softmax_dropout_fwd(b, h, lq, lk, _ptr(xx), _ptr(kl), int(bool(causal)),
                                   float(p), int(seed), int(offset), _ptr(y), _ptr(yd), _ptr(w))
    return y, yd, w


def softmax_dropout_bwd(y, dy_drop, mask, key_len, causal, p):
    yy, dd = _f64(y), _f64(dy_drop)
    b, h, lq, lk = yy.shape
    kl = _key_len(key_len)
    w = np.ascontiguousarray(np.asarray(mask, dtype=np.uint32))
    dx = np.empty_like(yy)
    _load().or_softmax_dropout_bwd(b, h, lq, lk, _ptr(yy), _ptr(dd), _ptr(w), _ptr(kl),
                                   int(bool(causal)), float(p), _ptr(dx))
    return dx


def cross_entropy_fwd(logits, target, eps=0.0, ignore_index=-100):
    """Returns (loss [rows], lse [rows]) for logits [rows, V] and int targets."""
    z = _f64(logits)
    rows, V = z.shape
    t = np.ascontiguousarray(np.asarray(target, dtype=np.int32))
    loss, lse = np.empty(rows), np.empty(rows)
    _load().or_cross_entropy_fwd(rows, V, _ptr(z), _ptr(t), float(eps), int(ignore_index),
                                 _ptr(loss), _ptr(lse))
    return loss, lse


def cross_entropy_bwd(logits, target, dloss=None, eps=0.0, ignore_index=-100):
    z = _f64(logits)
    rows, V = z.shape
    t = np.ascontiguousarray(np.asarray(target, dtype=np.int32))
    g = None if dloss is None else _f64(dloss)
    dz = np.empty_like(z)
    _load().or_cross_entropy_bwd(rows, V, _ptr(z), _ptr(t), _ptr(g), float(eps),
                                 int(ignore_index), _ptr(dz))
    return dz


def embedding_fwd(tokens, E, P, batch, seq, s, p, seed, offset):
    """Returns (y [batch*seq, H], mask words) of the embedding layer."""
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32)).ravel()
    e, pp = _f64(E), _f64(P)
    vocab, H = e.shape
    assert t.size == batch * seq and pp.shape[0] >= seq and pp.shape[1] == H
    y = np.empty((batch * seq, H))
    w = np.zeros(mask_words(y.size), dtype=np.uint32)
    _load().or_embedding_fwd(batch, seq, H, vocab, _ptr(t), _ptr(e), _ptr(pp), float(s),
                             float(p), int(seed), int(offset), _ptr(y), _ptr(w))
    return y, w


def embedding_bwd(tokens, dy, mask, vocab, s, p, dE=None):
    """dE [vocab, H] (float64) after adding the gradient of every token
    (starting from zeros, or from a copy of dE)."""
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32)).ravel()
    g = _f64(dy)
    T, H = g.shape
    out = np.zeros((vocab, H)) if dE is None else _f64(dE).copy()
    w = np.ascontiguousarray(np.asarray(mask, dtype=np.uint32))
    _load().or_embedding_bwd(T, H, vocab, _ptr(t), _ptr(g), _ptr(w), float(s), float(p),
                             _ptr(out))
    return out

