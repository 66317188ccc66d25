"""GPU parity: bias + reshape of Q, K, V, forward and backward, against the
FP64 oracle through the C ABI.  The forward is a bias add and a permutation,
the backward a permutation and a column sum: every element is compared, the
moved values exactly where the arithmetic allows (FP16 bias add rounds once),
the bias gradient within |err| <= 2e-3 + 2e-3*|ref| and bit-identical from
run to run.  Shapes: the four layer configurations and ragged ones (rows not
a multiple of the 128-row tile, columns not a multiple of the 64-column band)."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import Guarded, assert_close, dev, f64, require_gpu, tdtype
from transformer_layer_non_gb300 import ls_ops, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = [  # batch, seq, heads, head_dim, dtype
    (2, 16, 4, 16, "f32"),        # tiny layer
    (64, 64, 8, 64, "f16"),       # Transformer-base
    (8, 512, 12, 64, "f16"),      # BERT-base
    (4, 1024, 20, 64, "f16"),     # GPT-2-large
    (3, 37, 3, 24, "f16"),        # ragged: 111 rows, 216 columns
    (1, 1, 1, 8, "f32"),
    (5, 29, 2, 40, "f32"),
]


def _inputs(b, s, h, d, dtype, seed=0):
    qkv = synth.normal(seed, f"qkv{b}x{s}x{h}x{d}/x", (b * s, 3 * h * d), 0.0, 1.0, dtype)
    bias = synth.normal(seed, f"qkv{b}x{s}x{h}x{d}/bias", (3 * h * d,), 0.0, 0.02, dtype)
    dout = synth.normal(seed, f"qkv{b}x{s}x{h}x{d}/dout", (3, b, h, s, d), 0.0, 1.0, dtype)
    return qkv, bias, dout


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_forward_and_backward(case):
    require_gpu()
    b, s, h, d, dtype = case
    qkv, bias, dout = _inputs(b, s, h, d, dtype)
    out = Guarded((3, b, h, s, d), tdtype(qkv.dtype))
    ls_ops.ls_bias_reshape_qkv_fwd(out.t, dev(qkv), dev(bias), b, s, h)
    torch.cuda.synchronize()
    out.check()
    assert_close(f64(out.t), oracle.bias_reshape_qkv_fwd(qkv, bias, b, s, h, d), "q_k_v")

    rdq, rdb = oracle.bias_reshape_qkv_bwd(dout, b, s, h, d)
    ws = torch.empty(max(ls_ops.colreduce_workspace_bytes(b * s, 3 * h * d), 16),
                     dtype=torch.uint8, device="cuda").fill_(0xFF)
    results = []
    for _ in range(2):
        dq = Guarded((b * s, 3 * h * d), tdtype(qkv.dtype))
        db = Guarded((3 * h * d,), tdtype(qkv.dtype))
        ls_ops.ls_bias_reshape_qkv_bwd(dq.t, db.t, dev(dout), b, s, h, workspace=ws)
        torch.cuda.synchronize()
        dq.check()
        db.check()
        # The gradient moves without arithmetic: bit-exact.
        np.testing.assert_array_equal(f64(dq.t), rdq)
        assert_close(f64(db.t), rdb, "dbias")
        results.append(f64(db.t))
    np.testing.assert_array_equal(results[0], results[1])


def test_backward_without_bias_grad_and_empty_batch():
    require_gpu()
    b, s, h, d = 2, 8, 2, 16
    _, _, dout = _inputs(b, s, h, d, "f16", seed=3)
    dq = torch.empty((b * s, 3 * h * d), dtype=torch.float16, device="cuda")
    ls_ops.ls_bias_reshape_qkv_bwd(dq, None, dev(dout), b, s, h)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(f64(dq), oracle.bias_reshape_qkv_bwd(dout, b, s, h, d)[0])
    db = torch.full((3 * h * d,), 7.0, dtype=torch.float16, device="cuda")
    e = torch.empty((3, 0, h, s, d), dtype=torch.float16, device="cuda")
    ls_ops.ls_bias_reshape_qkv_bwd(dq, db, e, 0, s, h)
    torch.cuda.synchronize()
    assert (db == 0).all()
