"""The C-ABI library loads, exports every entry point that include/ls_ops.h
declares, and rejects bad arguments on the host before touching the GPU.

Only argument errors are exercised here: every call below returns before any
CUDA call, so this file runs on a machine without a GPU.  The pointers are
fake addresses that are never dereferenced.
"""
import ctypes
import os
import re
import subprocess

import pytest

from transformer_layer_non_gb300 import build as lsbuild
from transformer_layer_non_gb300 import ls_ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ls_ops.h")

A = 0x7F0000000000  # 16-byte aligned fake device addresses, far apart
B = A + (1 << 32)
C = A + (2 << 32)
D = A + (3 << 32)
E = A + (4 << 32)
F = A + (5 << 32)
G = A + (6 << 32)
H = A + (7 << 32)
I = A + (8 << 32)
S = None  # default stream


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ls_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return ls_ops.load()


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) == 27
    assert set(names) == set(ls_ops.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", lsbuild.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ls_[a-z0-9_]+)$", out, flags=re.M))
    assert set(names) <= exported
    # Nothing else leaks: the kernels and helpers are hidden.
    assert exported == set(names)
    for n in names:
        assert getattr(lib, n) is not None


def test_status_strings_and_version(lib):
    assert ls_ops.status_string(0) == "LS_OK"
    assert ls_ops.status_string(5) == "LS_ERR_CUDA"
    assert ls_ops.version() >= 10000


def test_workspace_query_is_shape_only(lib):
    # Partial rows depend on the shape only: one per 128 rows for the dropout
    # bias gradient, one per LayerNorm backward CTA for [dgamma | dbeta].
    assert ls_ops.colreduce_workspace_bytes(0, 768) == 0
    assert ls_ops.colreduce_workspace_bytes(4096, 7) == 0
    ws = ls_ops.colreduce_workspace_bytes(4096, 768)
    assert ws >= 32 * 768 * 4 and ws % 4 == 0
    assert ls_ops.colreduce_workspace_bytes(4096, 5120) >= 32 * 5120 * 4


def st(fn, *args):
    return getattr(ls_ops.load(), fn)(*args)


F16, F32 = ls_ops.LS_F16, ls_ops.LS_F32


def bdr_fwd(**kw):
    a = dict(dtype=F16, out=A, mask=B, x=C, bias=D, res=E, rows=4, cols=64, p=0.1, seed=0, off=0)
    a.update(kw)
    return st("ls_bias_dropout_residual_fwd", a["dtype"], a["out"], a["mask"], a["x"], a["bias"],
              a["res"], a["rows"], a["cols"], a["p"], a["seed"], a["off"], S)


def test_bdr_fwd_argument_errors(lib):
    assert bdr_fwd(out=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert "out is NULL" in ls_ops.last_error()
    assert bdr_fwd(x=C + 8) == ls_ops.LS_ERR_MISALIGNED
    assert bdr_fwd(cols=60) == ls_ops.LS_ERR_MISALIGNED
    assert bdr_fwd(cols=0) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bdr_fwd(rows=-1) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bdr_fwd(p=1.0) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bdr_fwd(p=-0.1) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bdr_fwd(p=float("nan")) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bdr_fwd(dtype=7) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bdr_fwd(cols=1 << 23) == ls_ops.LS_ERR_UNSUPPORTED_SHAPE
    # Partial overlap of the output with an input is rejected; exact aliasing is not.
    assert bdr_fwd(out=C + 16) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert "overlaps" in ls_ops.last_error()
    assert bdr_fwd(mask=C) == ls_ops.LS_ERR_INVALID_ARGUMENT  # mask inside x
    # rows == 0 is a no-op (nothing is enqueued), even with NULL pointers.
    assert bdr_fwd(rows=0, out=None, x=None) == ls_ops.LS_OK
    assert ls_ops.last_error() == ""


def test_dropout_bwd_argument_errors(lib):
    def bdr_bwd(dx=A, db=B, dout=C, mask=D, rows=256, cols=64, p=0.1, ws=E, wsb=1 << 20):
        return st("ls_bias_dropout_residual_bwd", F16, dx, db, dout, mask, rows, cols, p, 0, 0,
                  ws, wsb, S)

    # 256 rows -> two 128-row partial sums of 64 FP32 columns = 512 bytes.
    assert ls_ops.colreduce_workspace_bytes(256, 64) >= 512
    assert bdr_bwd(ws=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bdr_bwd(wsb=508) == ls_ops.LS_ERR_WORKSPACE_TOO_SMALL
    assert bdr_bwd(dout=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bdr_bwd(db=C + 64) == ls_ops.LS_ERR_INVALID_ARGUMENT        # dbias inside dout
    assert bdr_bwd(ws=A + 32) == ls_ops.LS_ERR_INVALID_ARGUMENT        # workspace inside dx
    assert bdr_bwd(rows=0, db=None) == ls_ops.LS_OK
    # bias+ReLU+dropout needs the mask (it cannot be redrawn: it holds the ReLU pattern).
    assert st("ls_bias_relu_dropout_bwd", F16, A, B, C, None, 256, 64, 0.1, E, 1 << 20,
              S) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert st("ls_bias_relu_dropout_fwd", F16, A, None, C, D, 256, 64, 0.1, 0, 0,
              S) == ls_ops.LS_ERR_INVALID_ARGUMENT


def test_layernorm_argument_errors(lib):
    def ln_fwd(y=A, mean=B, rstd=C, x=D, g=E, b=F, rows=8, cols=768, eps=1e-5, dtype=F16):
        return st("ls_layernorm_fwd", dtype, y, mean, rstd, x, g, b, rows, cols, eps, S)

    assert ln_fwd(cols=16392) == ls_ops.LS_ERR_UNSUPPORTED_SHAPE
    assert ln_fwd(eps=-1.0) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert ln_fwd(eps=float("inf")) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert ln_fwd(g=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert ln_fwd(mean=B + 4) == ls_ops.LS_ERR_MISALIGNED
    assert ln_fwd(rows=0) == ls_ops.LS_OK

    def ln_bwd(dx=A, dg=B, db=C, dy=D, x=E, g=F, mean=G, rstd=H, rows=8, cols=768, ws=I,
               wsb=1 << 24):
        return st("ls_layernorm_bwd", F16, dx, dg, db, dy, x, g, mean, rstd, rows, cols, ws, wsb, S)

    assert ln_bwd(db=None) == ls_ops.LS_ERR_INVALID_ARGUMENT   # dgamma without dbeta
    assert ln_bwd(wsb=16) == ls_ops.LS_ERR_WORKSPACE_TOO_SMALL
    assert ln_bwd(mean=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert ln_bwd(dx=E + 16) == ls_ops.LS_ERR_INVALID_ARGUMENT  # dx partially over x


def test_softmax_argument_errors(lib):
    def sm(y=A, x=B, b=2, h=3, lq=5, lk=64, kl=C, causal=0):
        return st("ls_softmax_fwd", F16, y, x, b, h, lq, lk, kl, causal, S)

    assert sm(lk=60) == ls_ops.LS_ERR_MISALIGNED
    assert sm(lk=0) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert sm(lk=(1 << 20) + 8) == ls_ops.LS_ERR_UNSUPPORTED_SHAPE
    assert sm(kl=C + 2) == ls_ops.LS_ERR_MISALIGNED
    assert sm(b=-1) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert sm(x=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert sm(y=B + 128) == ls_ops.LS_ERR_INVALID_ARGUMENT      # partial overlap
    assert sm(h=0) == ls_ops.LS_OK                                 # empty: no-op
    assert st("ls_softmax_bwd", F16, A, B, None, 2, 3, 5, 64, None, 0,
              S) == ls_ops.LS_ERR_INVALID_ARGUMENT


def test_error_message_is_per_thread(lib):
    import threading

    assert bdr_fwd(out=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    seen = {}

    def other():
        seen["msg"] = ls_ops.last_error()

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert seen["msg"] == ""
    assert "out is NULL" in ls_ops.last_error()


def test_adam_update_argument_errors(lib):
    def adam(p=A, g=B, m=C, v=D, n=1000, lr=1e-3, b1=0.9, b2=0.999, eps=1e-8, wd=0.0, step=1,
             gs=1.0, dtype=F16):
        return st("ls_adam_update", dtype, p, g, m, v, n, lr, b1, b2, eps, wd, step, gs, S)

    assert adam(n=-1) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert adam(step=0) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert adam(b1=1.0) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert adam(b2=-0.1) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert adam(lr=float("nan")) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert adam(eps=-1e-8) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert adam(wd=float("inf")) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert adam(gs=float("inf")) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert adam(dtype=3) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert adam(m=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert adam(v=D + 4) == ls_ops.LS_ERR_MISALIGNED
    assert adam(g=A) == ls_ops.LS_ERR_INVALID_ARGUMENT                 # grad is param
    assert adam(m=A + 512) == ls_ops.LS_ERR_INVALID_ARGUMENT           # exp_avg inside param
    assert adam(g=C + 16) == ls_ops.LS_ERR_INVALID_ARGUMENT            # grad inside exp_avg
    assert adam(n=1 << 47) == ls_ops.LS_ERR_UNSUPPORTED_SHAPE
    assert adam(n=0, p=None, g=None) == ls_ops.LS_OK
    assert ls_ops.last_error() == ""


def test_bias_reshape_qkv_argument_errors(lib):
    def fwd(out=A, qkv=B, bias=C, b=2, s=16, h=4, d=64, dtype=F16):
        return st("ls_bias_reshape_qkv_fwd", dtype, out, qkv, bias, b, s, h, d, S)

    def bwd(dqkv=A, db=B, dout=C, b=2, s=16, h=4, d=64, ws=D, wsb=1 << 20):
        return st("ls_bias_reshape_qkv_bwd", F16, dqkv, db, dout, b, s, h, d, ws, wsb, S)

    assert fwd(d=60) == ls_ops.LS_ERR_MISALIGNED
    assert fwd(d=0) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert fwd(b=-1) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert fwd(bias=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert fwd(out=B) == ls_ops.LS_ERR_INVALID_ARGUMENT          # no in-place reshape
    assert fwd(qkv=B + 8) == ls_ops.LS_ERR_MISALIGNED
    assert fwd(h=1 << 20) == ls_ops.LS_ERR_UNSUPPORTED_SHAPE
    assert fwd(b=0, out=None) == ls_ops.LS_OK
    # 32 rows of 3 x 4 x 64 columns -> one 128-row partial row of 768 FP32 sums.
    assert bwd(wsb=768 * 4 - 4) == ls_ops.LS_ERR_WORKSPACE_TOO_SMALL
    assert bwd(ws=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bwd(dout=A) == ls_ops.LS_ERR_INVALID_ARGUMENT         # no in-place reshape
    assert ls_ops.colreduce_workspace_bytes(32, 768) >= 768 * 4


def test_softmax_dropout_argument_errors(lib):
    def fwd(y=A, yd=B, m=C, x=D, b=2, h=2, lq=4, lk=64, kl=None, p=0.1):
        return st("ls_softmax_dropout_fwd", F16, y, yd, m, x, b, h, lq, lk, kl, 0, p, 0, 0, S)

    def bwd(dx=A, y=B, dyd=C, m=D, b=2, h=2, lq=4, lk=64, p=0.1):
        return st("ls_softmax_dropout_bwd", F16, dx, y, dyd, m, b, h, lq, lk, None, 0, p, S)

    assert fwd(p=1.0) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert fwd(m=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert fwd(yd=A) == ls_ops.LS_ERR_INVALID_ARGUMENT          # y_drop is y
    assert fwd(m=D + 64) == ls_ops.LS_ERR_INVALID_ARGUMENT      # mask inside x
    assert fwd(lk=60) == ls_ops.LS_ERR_MISALIGNED
    assert fwd(kl=E + 2) == ls_ops.LS_ERR_MISALIGNED
    assert fwd(b=0, y=None) == ls_ops.LS_OK
    assert bwd(p=-0.5) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bwd(m=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bwd(dx=B + 16) == ls_ops.LS_ERR_INVALID_ARGUMENT     # dx partly over y
    assert bwd(lq=0) == ls_ops.LS_OK


def test_cross_entropy_argument_errors(lib):
    def fwd(loss=A, lse=B, z=C, t=D, rows=4, V=64, eps=0.0, dtype=F16):
        return st("ls_cross_entropy_fwd", dtype, loss, lse, z, t, rows, V, eps, -100, S)

    def bwd(dz=A, z=B, t=C, lse=D, g=E, rows=4, V=64, eps=0.1):
        return st("ls_cross_entropy_bwd", F16, dz, z, t, lse, g, rows, V, eps, -100, S)

    assert fwd(V=60) == ls_ops.LS_ERR_MISALIGNED
    assert fwd(V=0) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert fwd(eps=1.0) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert fwd(t=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert fwd(t=D + 2) == ls_ops.LS_ERR_MISALIGNED
    assert fwd(lse=A) == ls_ops.LS_ERR_INVALID_ARGUMENT          # lse is loss
    assert fwd(rows=0, loss=None) == ls_ops.LS_OK
    assert bwd(lse=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bwd(dz=B + 16) == ls_ops.LS_ERR_INVALID_ARGUMENT       # dlogits partly over logits
    assert bwd(rows=-1) == ls_ops.LS_ERR_INVALID_ARGUMENT


def test_embedding_argument_errors(lib):
    def fwd(y=A, m=B, tok=C, E=D, P=E, b=2, s=16, h=64, v=100, mp=16, p=0.1):
        return st("ls_embedding_fwd", F16, y, m, tok, E, P, b, s, h, v, mp, 1.0, p, 0, 0, S)

    def bwd(dE=A, dy=B, m=C, tok=D, b=2, s=16, h=64, v=100, ws=E, wsb=1 << 20):
        return st("ls_embedding_bwd", F16, dE, dy, m, tok, b, s, h, v, 1.0, 0.1, 1, ws, wsb, S)

    assert ls_ops.embedding_workspace_bytes(32) == 0
    assert fwd(h=60) == ls_ops.LS_ERR_MISALIGNED
    assert fwd(mp=8) == ls_ops.LS_ERR_INVALID_ARGUMENT           # positions shorter than seq
    assert fwd(tok=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert fwd(tok=C + 2) == ls_ops.LS_ERR_MISALIGNED
    assert fwd(p=1.5) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert fwd(y=D) == ls_ops.LS_ERR_INVALID_ARGUMENT            # y over the token table
    assert fwd(b=0, y=None) == ls_ops.LS_OK
    # no workspace is needed: a NULL one gets past to the later checks
    assert bwd(ws=None, wsb=0, tok=D + 2) == ls_ops.LS_ERR_MISALIGNED
    assert bwd(m=None) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert bwd(b=1024, s=17) == ls_ops.LS_ERR_UNSUPPORTED_SHAPE   # > 16384 tokens in one call
    assert bwd(tok=A + 64) == ls_ops.LS_ERR_INVALID_ARGUMENT      # tokens inside dE


def test_selftest_argument_errors(lib):
    assert st("ls_selftest_wait_timeout", 0, S) == ls_ops.LS_ERR_INVALID_ARGUMENT
    assert st("ls_selftest_wait_timeout", (1 << 19) + 1, S) == ls_ops.LS_ERR_INVALID_ARGUMENT


def test_reduction_stream_default_and_empty_join(lib):
    # Restoring the default and joining with nothing forked make no CUDA call.
    assert lib.ls_set_reduction_stream(None) == ls_ops.LS_OK
    assert lib.ls_join_reductions(None) == ls_ops.LS_OK
    assert lib.ls_join_reductions(A) == ls_ops.LS_OK


def test_noalloc_scratch_size_matches_the_header():
    import re

    from transformer_layer_non_gb300 import ls_ops

    hdr = open(os.path.join(ROOT, "include", "ls_ops.h")).read()
    m = re.search(r"#define LS_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", hdr)
    assert m, "LS_NOALLOC_SCRATCH_BYTES not found in the header"
    assert ls_ops.LS_NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
