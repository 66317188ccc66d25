"""Thin Python binding of the ``ls_ops`` C ABI (``include/ls_ops.h``).

Each function has the C entry point's name and argument order, takes torch
CUDA tensors (or raw integers for pointers), and only marshals arguments:
every step of every operator runs in the CUDA library.  There is no fallback:
if the library cannot be built or loaded, importing this module's functions
raises.  Work is enqueued on ``stream`` (default: torch's current stream) and
nothing is synchronised.

Status codes other than ``LS_OK`` raise :class:`LsError` carrying the code
and the library's message.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

LS_OK = 0
LS_ERR_INVALID_ARGUMENT = 1
LS_ERR_MISALIGNED = 2
LS_ERR_UNSUPPORTED_SHAPE = 3
LS_ERR_WORKSPACE_TOO_SMALL = 4
LS_ERR_CUDA = 5

LS_F32 = 0
LS_F16 = 1

# Size of the scratch array behind ls_layernorm_bwd_noalloc (include/ls_ops.h).
LS_NOALLOC_SCRATCH_BYTES = 8 << 20

# Every entry point declared in include/ls_ops.h.
EXPORTS = (
    "ls_status_string", "ls_last_error", "ls_version", "ls_colreduce_workspace_bytes",
    "ls_bias_dropout_residual_fwd", "ls_bias_dropout_residual_bwd",
    "ls_bias_relu_dropout_fwd", "ls_bias_relu_dropout_bwd",
    "ls_layernorm_fwd", "ls_layernorm_bwd", "ls_softmax_fwd", "ls_softmax_bwd",
    "ls_layernorm_bwd_noalloc", "ls_check_device_errors", "ls_adam_update",
    "ls_bias_reshape_qkv_fwd", "ls_bias_reshape_qkv_bwd",
    "ls_softmax_dropout_fwd", "ls_softmax_dropout_bwd",
    "ls_cross_entropy_fwd", "ls_cross_entropy_bwd",
    "ls_embedding_fwd", "ls_embedding_bwd", "ls_embedding_workspace_bytes",
    "ls_selftest_wait_timeout", "ls_set_reduction_stream", "ls_join_reductions",
)


class LsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_F32 = ctypes.c_float
_INT = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "ls_status_string": (ctypes.c_char_p, [_INT]),
    "ls_last_error": (ctypes.c_char_p, []),
    "ls_version": (_INT, []),
    "ls_colreduce_workspace_bytes": (_SZ, [_I64, _I64]),
    "ls_check_device_errors": (_INT, [ctypes.POINTER(ctypes.c_uint32)]),
    "ls_bias_dropout_residual_fwd": (_INT, [_INT, _P, _P, _P, _P, _P, _I64, _I64, _F32, _U64, _U64, _P]),
    "ls_bias_dropout_residual_bwd": (_INT, [_INT, _P, _P, _P, _P, _I64, _I64, _F32, _U64, _U64, _P, _SZ, _P]),
    "ls_bias_relu_dropout_fwd": (_INT, [_INT, _P, _P, _P, _P, _I64, _I64, _F32, _U64, _U64, _P]),
    "ls_bias_relu_dropout_bwd": (_INT, [_INT, _P, _P, _P, _P, _I64, _I64, _F32, _P, _SZ, _P]),
    "ls_layernorm_fwd": (_INT, [_INT, _P, _P, _P, _P, _P, _P, _I64, _I64, _F32, _P]),
    "ls_layernorm_bwd": (_INT, [_INT, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P]),
    "ls_layernorm_bwd_noalloc": (_INT, [_INT, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P]),
    "ls_softmax_fwd": (_INT, [_INT, _P, _P, _I64, _I64, _I64, _I64, _P, _INT, _P]),
    "ls_softmax_bwd": (_INT, [_INT, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _INT, _P]),
    "ls_selftest_wait_timeout": (_INT, [ctypes.c_uint32, _P]),
    "ls_set_reduction_stream": (_INT, [_P]),
    "ls_join_reductions": (_INT, [_P]),
    "ls_embedding_fwd": (_INT, [_INT, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _F32,
                                _F32, _U64, _U64, _P]),
    "ls_embedding_bwd": (_INT, [_INT, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _F32, _F32, _INT,
                                _P, _SZ, _P]),
    "ls_embedding_workspace_bytes": (_SZ, [_I64]),
    "ls_cross_entropy_fwd": (_INT, [_INT, _P, _P, _P, _P, _I64, _I64, _F32, ctypes.c_int32, _P]),
    "ls_cross_entropy_bwd": (_INT, [_INT, _P, _P, _P, _P, _P, _I64, _I64, _F32, ctypes.c_int32,
                                    _P]),
    "ls_softmax_dropout_fwd": (_INT, [_INT, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _INT,
                                      _F32, _U64, _U64, _P]),
    "ls_softmax_dropout_bwd": (_INT, [_INT, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _INT,
                                      _F32, _P]),
    "ls_bias_reshape_qkv_fwd": (_INT, [_INT, _P, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "ls_bias_reshape_qkv_bwd": (_INT, [_INT, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _SZ, _P]),
    "ls_adam_update": (_INT, [_INT, _P, _P, _P, _P, _I64, _F32, _F32, _F32, _F32, _F32, _I64,
                              _F32, _P]),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_needed: bool = True):
    """Load libls_ops.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_needed else _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libls_ops.so not found at {path}; build it with "
                           "`python -m transformer_layer_non_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().ls_status_string(status).decode()


def last_error() -> str:
    return load().ls_last_error().decode()


def version() -> int:
    return load().ls_version()


def colreduce_workspace_bytes(rows: int, cols: int) -> int:
    return int(load().ls_colreduce_workspace_bytes(rows, cols))


def new_workspace(shapes, device="cuda"):
    """A workspace large enough for the backward calls with a column
    reduction on every [rows, cols] in `shapes`."""
    import torch

    n = max([colreduce_workspace_bytes(r, c) for r, c in shapes] + [256])
    return torch.zeros(n, dtype=torch.uint8, device=device)


LS_DEVERR_WAIT_TIMEOUT = 1


def check_device_errors() -> int:
    """Synchronise the current device and return (and clear) the library's
    device-side failure flags (0 = none)."""
    v = ctypes.c_uint32(0)
    _check(load().ls_check_device_errors(ctypes.byref(v)))
    return int(v.value)


def selftest_wait_timeout(polls: int = 1024, stream=None):
    """Enqueue the bounded-wait failure self-test (see include/ls_ops.h)."""
    _check(load().ls_selftest_wait_timeout(polls, _stream(stream)))


def set_reduction_stream(stream):
    """Fork the column reductions of the backward calls made from this thread
    onto `stream` (a torch.cuda.Stream or a raw handle); None restores the
    default.  See ls_set_reduction_stream in include/ls_ops.h."""
    h = None if stream is None else (stream if isinstance(stream, int) else stream.cuda_stream)
    _check(load().ls_set_reduction_stream(h))


def join_reductions(stream=None):
    """Order `stream` (default: the current stream) after every forked
    reduction; the gradients are ready from there on."""
    _check(load().ls_join_reductions(_stream(stream)))


def _check(status: int):
    if status != LS_OK:
        raise LsError(status, last_error())


# --- argument marshalling -------------------------------------------------
def _ptr(t) -> Optional[int]:
    """Device address of a tensor (or an int address, or None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float16:
        return LS_F16
    if t.dtype == torch.float32:
        return LS_F32
    raise TypeError(f"unsupported storage dtype {t.dtype}; use float16 or float32")


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _rows_cols(t):
    cols = t.shape[-1]
    return t.numel() // cols if cols else 0, cols


def _nbytes(ws) -> int:
    return 0 if ws is None else ws.numel() * ws.element_size()


# --- operators --------------------------------------------------------------
def ls_bias_dropout_residual_fwd(out, mask_bits, x, bias, residual, p: float, seed: int,
                                 offset: int, stream=None):
    rows, cols = _rows_cols(x)
    _check(load().ls_bias_dropout_residual_fwd(
        _dtype_code(x), _ptr(out), _ptr(mask_bits), _ptr(x), _ptr(bias), _ptr(residual),
        rows, cols, p, seed, offset, _stream(stream)))


def ls_bias_dropout_residual_bwd(dx, dbias, dout, mask_bits, p: float, seed: int = 0,
                                 offset: int = 0, workspace=None, stream=None):
    rows, cols = _rows_cols(dout)
    _check(load().ls_bias_dropout_residual_bwd(
        _dtype_code(dout), _ptr(dx), _ptr(dbias), _ptr(dout), _ptr(mask_bits), rows, cols, p,
        seed, offset, _ptr(workspace), _nbytes(workspace), _stream(stream)))


def ls_bias_relu_dropout_fwd(out, mask_bits, x, bias, p: float, seed: int, offset: int,
                             stream=None):
    rows, cols = _rows_cols(x)
    _check(load().ls_bias_relu_dropout_fwd(
        _dtype_code(x), _ptr(out), _ptr(mask_bits), _ptr(x), _ptr(bias), rows, cols, p, seed,
        offset, _stream(stream)))


def ls_bias_relu_dropout_bwd(dx, dbias, dout, mask_bits, p: float, workspace=None, stream=None):
    rows, cols = _rows_cols(dout)
    _check(load().ls_bias_relu_dropout_bwd(
        _dtype_code(dout), _ptr(dx), _ptr(dbias), _ptr(dout), _ptr(mask_bits), rows, cols, p,
        _ptr(workspace), _nbytes(workspace), _stream(stream)))


def ls_layernorm_fwd(y, mean, rstd, x, gamma, beta, eps: float = 1e-5, stream=None):
    rows, cols = _rows_cols(x)
    _check(load().ls_layernorm_fwd(
        _dtype_code(x), _ptr(y), _ptr(mean), _ptr(rstd), _ptr(x), _ptr(gamma), _ptr(beta),
        rows, cols, eps, _stream(stream)))


def ls_layernorm_bwd(dx, dgamma, dbeta, dy, x, gamma, mean, rstd, workspace=None, stream=None):
    rows, cols = _rows_cols(x)
    _check(load().ls_layernorm_bwd(
        _dtype_code(x), _ptr(dx), _ptr(dgamma), _ptr(dbeta), _ptr(dy), _ptr(x), _ptr(gamma),
        _ptr(mean), _ptr(rstd), rows, cols, _ptr(workspace), _nbytes(workspace),
        _stream(stream)))


def ls_layernorm_bwd_noalloc(dx, dgamma, dbeta, dy, x, gamma, mean, rstd, stream=None):
    """ls_layernorm_bwd without a workspace argument: the gamma/beta partial
    sums go to the library's built-in device scratch (for callers that cannot
    allocate device memory).  Calls that overlap on the GPU must not be issued."""
    rows, cols = _rows_cols(x)
    _check(load().ls_layernorm_bwd_noalloc(
        _dtype_code(x), _ptr(dx), _ptr(dgamma), _ptr(dbeta), _ptr(dy), _ptr(x), _ptr(gamma),
        _ptr(mean), _ptr(rstd), rows, cols, _stream(stream)))


def ls_softmax_fwd(y, x, key_len=None, causal: bool = False, stream=None):
    """x, y: [batch, heads, q_len, k_len]; key_len: int32 [batch] on the device or None."""
    b, h, lq, lk = x.shape
    _check(load().ls_softmax_fwd(_dtype_code(x), _ptr(y), _ptr(x), b, h, lq, lk, _ptr(key_len),
                                 int(bool(causal)), _stream(stream)))


def ls_softmax_bwd(dx, y, dy, key_len=None, causal: bool = False, stream=None):
    b, h, lq, lk = y.shape
    _check(load().ls_softmax_bwd(_dtype_code(y), _ptr(dx), _ptr(y), _ptr(dy), b, h, lq, lk,
                                 _ptr(key_len), int(bool(causal)), _stream(stream)))


def ls_adam_update(param, grad, exp_avg, exp_avg_sq, lr: float, beta1: float, beta2: float,
                   eps: float, weight_decay: float, step: int, grad_scale: float = 1.0,
                   stream=None):
    """One trainer update of a flat workspace, in place: param and grad in the
    storage dtype, exp_avg and exp_avg_sq FP32, all with param.numel() elements."""
    n = param.numel()
    for t in (grad, exp_avg, exp_avg_sq):
        if t.numel() != n:
            raise ValueError("param, grad, exp_avg and exp_avg_sq must have the same size")
    _check(load().ls_adam_update(_dtype_code(param), _ptr(param), _ptr(grad), _ptr(exp_avg),
                                 _ptr(exp_avg_sq), n, lr, beta1, beta2, eps, weight_decay,
                                 int(step), grad_scale, _stream(stream)))


def ls_bias_reshape_qkv_fwd(q_k_v, qkv, bias, batch: int, seq: int, heads: int,
                            stream=None):
    """qkv [batch*seq, 3*H] + bias [3*H] -> q_k_v [3, batch, heads, seq, H/heads]."""
    d = q_k_v.shape[-1]
    _check(load().ls_bias_reshape_qkv_fwd(_dtype_code(qkv), _ptr(q_k_v), _ptr(qkv), _ptr(bias),
                                          batch, seq, heads, d, _stream(stream)))


def ls_bias_reshape_qkv_bwd(dqkv, dbias, dq_k_v, batch: int, seq: int, heads: int,
                            workspace=None, stream=None):
    """dq_k_v [3, batch, heads, seq, d] -> dqkv [batch*seq, 3*H] and dbias [3*H]."""
    d = dq_k_v.shape[-1]
    _check(load().ls_bias_reshape_qkv_bwd(_dtype_code(dq_k_v), _ptr(dqkv), _ptr(dbias),
                                          _ptr(dq_k_v), batch, seq, heads, d, _ptr(workspace),
                                          _nbytes(workspace), _stream(stream)))


def ls_softmax_dropout_fwd(y, y_drop, mask_bits, x, key_len=None, causal: bool = False,
                           p: float = 0.1, seed: int = 0, offset: int = 0, stream=None):
    """Softmax of x [batch, heads, q_len, k_len] into y, then dropout on the
    probabilities into y_drop with its bits in mask_bits (int32 words)."""
    b, h, lq, lk = x.shape
    _check(load().ls_softmax_dropout_fwd(_dtype_code(x), _ptr(y), _ptr(y_drop), _ptr(mask_bits),
                                         _ptr(x), b, h, lq, lk, _ptr(key_len), int(bool(causal)),
                                         p, seed, offset, _stream(stream)))


def ls_softmax_dropout_bwd(dx, y, dy_drop, mask_bits, key_len=None, causal: bool = False,
                           p: float = 0.1, stream=None):
    b, h, lq, lk = y.shape
    _check(load().ls_softmax_dropout_bwd(_dtype_code(y), _ptr(dx), _ptr(y), _ptr(dy_drop),
                                         _ptr(mask_bits), b, h, lq, lk, _ptr(key_len),
                                         int(bool(causal)), p, _stream(stream)))


def ls_cross_entropy_fwd(loss, lse, logits, target, label_smoothing: float = 0.0,
                         ignore_index: int = -100, stream=None):
    """Per-row loss (FP32 [rows]) and lse (FP32 [rows] or None) of logits
    [rows, vocab] against int32 targets [rows]."""
    rows, vocab = logits.shape
    _check(load().ls_cross_entropy_fwd(_dtype_code(logits), _ptr(loss), _ptr(lse), _ptr(logits),
                                       _ptr(target), rows, vocab, label_smoothing, ignore_index,
                                       _stream(stream)))


def ls_cross_entropy_bwd(dlogits, logits, target, lse, dloss=None, label_smoothing: float = 0.0,
                         ignore_index: int = -100, stream=None):
    rows, vocab = logits.shape
    _check(load().ls_cross_entropy_bwd(_dtype_code(logits), _ptr(dlogits), _ptr(logits),
                                       _ptr(target), _ptr(lse), _ptr(dloss), rows, vocab,
                                       label_smoothing, ignore_index, _stream(stream)))


def ls_embedding_fwd(y, mask_bits, tokens, token_table, pos_table, batch: int, seq: int,
                     scale: float, p: float, seed: int = 0, offset: int = 0, stream=None):
    """y [batch*seq, H] = Dropout(scale * E[tokens] + P[positions])."""
    vocab, hidden = token_table.shape
    _check(load().ls_embedding_fwd(_dtype_code(token_table), _ptr(y), _ptr(mask_bits),
                                   _ptr(tokens), _ptr(token_table), _ptr(pos_table), batch, seq,
                                   hidden, vocab, pos_table.shape[0], scale, p, seed, offset,
                                   _stream(stream)))


def embedding_workspace_bytes(tokens: int) -> int:
    return int(load().ls_embedding_workspace_bytes(tokens))


def ls_embedding_bwd(d_token_table, dy, mask_bits, tokens, batch: int, seq: int, scale: float,
                     p: float, deterministic: bool = True, workspace=None, stream=None):
    """Adds the token-table gradient (FP32 [vocab, H]) of this batch into
    d_token_table: deterministically (each id's sum in an order fixed by the
    ids) or with float atomics.  No workspace is needed."""
    vocab, hidden = d_token_table.shape
    _check(load().ls_embedding_bwd(_dtype_code(dy), _ptr(d_token_table), _ptr(dy),
                                   _ptr(mask_bits), _ptr(tokens), batch, seq, hidden, vocab,
                                   scale, p, int(bool(deterministic)), _ptr(workspace),
                                   _nbytes(workspace), _stream(stream)))

