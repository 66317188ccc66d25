"""ls_layernorm_bwd_noalloc: the LayerNorm backward for callers that cannot
allocate device memory (and so cannot pass a workspace).  Its gamma/beta
partial sums live in a scratch array built into the library.

Checked through the C ABI against ls_layernorm_bwd with a caller workspace,
within the parity tolerance |err| <= 2e-3 + 2e-3*|ref|, on two calls in a row
(the second call finds the first call's leftovers in the shared scratch).
This file is collected last and also passes when run on its own."""
import numpy as np
import pytest

import oracle
from transformer_layer_non_gb300 import ls_ops, synth
from tests.gpu_util import assert_close, dev, f64, require_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EPS = 1e-5


def _case(seed, rows, cols):
    x = synth.normal(seed, f"na/x{cols}", (rows, cols), 0.0, 1.0, "f16")
    dy = synth.normal(seed, f"na/dy{cols}", (rows, cols), 0.0, 1.0, "f16")
    g = synth.normal(seed, f"na/g{cols}", (cols,), 1.0, 0.1, "f16")
    _, mean, rstd = oracle.layernorm_fwd(x, g, np.zeros_like(g), EPS)
    return dev(x), dev(dy), dev(g), dev(mean.astype(np.float32)), dev(rstd.astype(np.float32))


def _with_workspace(x, dy, g, mean, rstd):
    rows, cols = x.shape
    dx, dg, db = torch.empty_like(x), torch.empty_like(g), torch.empty_like(g)
    ws = ls_ops.new_workspace([(rows, cols)])
    ls_ops.ls_layernorm_bwd(dx, dg, db, dy, x, g, mean, rstd, workspace=ws)
    return dx, dg, db


def _no_alloc(x, dy, g, mean, rstd):
    dx, dg, db = torch.empty_like(x), torch.empty_like(g), torch.empty_like(g)
    ls_ops.ls_layernorm_bwd_noalloc(dx, dg, db, dy, x, g, mean, rstd)
    return dx, dg, db


def test_no_alloc_matches_workspace_entry_point_on_two_calls():
    require_gpu()
    # GPT-2-large width, then BERT-base width: the second call reuses the
    # scratch the first one left behind.
    for seed, rows, cols in [(1, 4096, 1280), (2, 4096, 768)]:
        args = _case(seed, rows, cols)
        got = _no_alloc(*args)
        ref = _with_workspace(*args)
        torch.cuda.synchronize()
        for name, a, b in zip(("dx", "dgamma", "dbeta"), got, ref):
            assert_close(f64(a), f64(b), f"no-alloc {name} ({rows}x{cols})")


def test_no_alloc_rejects_shapes_beyond_its_scratch():
    require_gpu()
    lib = ls_ops.load()
    fake = 0x7F0000000000  # never dereferenced: the call is rejected first
    st = lib.ls_layernorm_bwd_noalloc(ls_ops.LS_F16, fake, fake + (1 << 32), fake + (2 << 32),
                                      fake + (3 << 32), fake + (4 << 32), fake + (5 << 32),
                                      fake + (6 << 32), fake + (7 << 32), 1 << 20, 16384, None)
    assert st == ls_ops.LS_ERR_UNSUPPORTED_SHAPE
    assert "scratch" in ls_ops.last_error()
