"""GPU parity: fused bias+dropout+residual and bias+ReLU+dropout against the
FP64 oracle.  Masks (keep bits; ReLU-and-keep bits) must match bit for bit;
values within |err| <= 2e-3 + 2e-3*|ref|.  The layer configurations run at
their full sizes, every element compared."""
import numpy as np
import pytest

import oracle
from transformer_layer_non_gb300 import ls_ops, synth
from tests.gpu_util import Guarded, assert_close, dev, f64, mask_words_of, require_gpu, tdtype

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LAYERS = ["tiny", "transformer-base", "bert-base", "gpt2-large"]
SEED, OFF_ATTN, OFF_FFN1 = 0, 11, 12


def _mask_buf(n):
    return Guarded(((n + 31) // 32,), torch.int32)


def _ws(rows, cols):
    return torch.empty(max(ls_ops.colreduce_workspace_bytes(rows, cols), 16), dtype=torch.uint8,
                       device="cuda").fill_(0xFF)  # garbage: the workspace needs no init


def run_bdr_fwd(x, bias, res, p, seed, off):
    rows, cols = x.shape
    out = Guarded(x.shape, tdtype(x.dtype))
    mask = _mask_buf(rows * cols)
    ls_ops.ls_bias_dropout_residual_fwd(out.t, mask.t, dev(x), dev(bias), dev(res), p, seed, off)
    torch.cuda.synchronize()
    out.check()
    mask.check()
    return f64(out.t), mask_words_of(mask.t)


def run_dropout_bwd(relu, dout, mask_words, p, seed=0, off=0, with_mask=True):
    rows, cols = dout.shape
    dx = Guarded(dout.shape, tdtype(dout.dtype))
    db = Guarded((cols,), tdtype(dout.dtype))
    m = dev(mask_words.view(np.int32)) if with_mask else None
    ws = _ws(rows, cols)
    if relu:
        ls_ops.ls_bias_relu_dropout_bwd(dx.t, db.t, dev(dout), m, p, workspace=ws)
    else:
        ls_ops.ls_bias_dropout_residual_bwd(dx.t, db.t, dev(dout), m, p, seed, off, workspace=ws)
    torch.cuda.synchronize()
    dx.check()
    db.check()
    return f64(dx.t), f64(db.t)


@pytest.mark.parametrize("name", LAYERS)
def test_bias_dropout_residual_layer(name):
    require_gpu()
    L = synth.LAYERS[name]
    d = synth.layer_inputs(L, SEED, which={"attn_x", "attn_res", "attn_bias", "attn_dout"})
    out, mask = run_bdr_fwd(d["attn_x"], d["attn_bias"], d["attn_res"], L.p, SEED, OFF_ATTN)
    ref, ref_mask = oracle.bias_dropout_residual_fwd(d["attn_x"], d["attn_bias"], d["attn_res"],
                                                     L.p, SEED, OFF_ATTN)
    np.testing.assert_array_equal(mask, ref_mask)
    assert_close(out, ref, f"{name} bdr fwd")
    dx, db = run_dropout_bwd(False, d["attn_dout"], mask, L.p)
    rdx, rdb = oracle.bias_dropout_residual_bwd(d["attn_dout"], ref_mask, L.p)
    assert_close(dx, rdx, f"{name} bdr bwd dx")
    assert_close(db, rdb, f"{name} bdr bwd dbias")
    # Without the saved mask the bits are drawn again from (seed, offset).
    dx2, db2 = run_dropout_bwd(False, d["attn_dout"], mask, L.p, SEED, OFF_ATTN, with_mask=False)
    np.testing.assert_array_equal(dx2, dx)
    np.testing.assert_array_equal(db2, db)


@pytest.mark.parametrize("name", LAYERS)
def test_bias_relu_dropout_layer(name):
    require_gpu()
    L = synth.LAYERS[name]
    d = synth.layer_inputs(L, SEED, which={"ffn1_x", "ffn1_bias", "ffn1_dout"})
    x, bias = d["ffn1_x"], d["ffn1_bias"]
    rows, cols = x.shape
    out = Guarded(x.shape, tdtype(x.dtype))
    mask = _mask_buf(rows * cols)
    ls_ops.ls_bias_relu_dropout_fwd(out.t, mask.t, dev(x), dev(bias), L.p, SEED, OFF_FFN1)
    torch.cuda.synchronize()
    out.check()
    mask.check()
    ref, ref_mask = oracle.bias_relu_dropout_fwd(x, bias, L.p, SEED, OFF_FFN1)
    np.testing.assert_array_equal(mask_words_of(mask.t), ref_mask)
    assert_close(f64(out.t), ref, f"{name} brd fwd")
    dx, db = run_dropout_bwd(True, d["ffn1_dout"], ref_mask, L.p)
    rdx, rdb = oracle.bias_relu_dropout_bwd(d["ffn1_dout"], ref_mask, L.p)
    assert_close(dx, rdx, f"{name} brd bwd dx")
    assert_close(db, rdb, f"{name} brd bwd dbias")


RAGGED = [(1, 8), (3, 24), (37, 72), (129, 264), (300, 2056), (257, 520)]


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("shape", RAGGED)
@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
def test_ragged_shapes(dtype, shape, p):
    # Row counts that are not a multiple of the tile, column counts that leave a
    # partial column band, and element counts whose last mask word is partial.
    require_gpu()
    rows, cols = shape
    x = synth.normal(3, "rag/x", shape, 0.0, 1.0, dtype)
    r = synth.normal(3, "rag/r", shape, 0.0, 1.0, dtype)
    b = synth.normal(3, "rag/b", (cols,), 0.0, 0.02, dtype)
    g = synth.normal(3, "rag/g", shape, 0.0, 1.0, dtype)
    seed, off = 0x1234_5678_9ABC_DEF0, 0xFEDC_BA98_0000_0001  # high words in use
    out, mask = run_bdr_fwd(x, b, r, p, seed, off)
    ref, ref_mask = oracle.bias_dropout_residual_fwd(x, b, r, p, seed, off)
    np.testing.assert_array_equal(mask, ref_mask)  # includes the zeroed tail bits
    assert_close(out, ref, "ragged bdr fwd")
    dx, db = run_dropout_bwd(False, g, mask, p, seed, off, with_mask=False)
    rdx, rdb = oracle.bias_dropout_residual_bwd(g, None, p, seed, off)
    assert_close(dx, rdx, "ragged bdr bwd dx")
    assert_close(db, rdb, "ragged bdr bwd dbias")
    # bias+ReLU+dropout on the same shape
    o2 = Guarded(shape, tdtype(x.dtype))
    m2 = _mask_buf(rows * cols)
    ls_ops.ls_bias_relu_dropout_fwd(o2.t, m2.t, dev(x), dev(b), p, seed, off)
    torch.cuda.synchronize()
    o2.check()
    m2.check()
    ref2, ref_m2 = oracle.bias_relu_dropout_fwd(x, b, p, seed, off)
    np.testing.assert_array_equal(mask_words_of(m2.t), ref_m2)
    assert_close(f64(o2.t), ref2, "ragged brd fwd")
    dx2, db2 = run_dropout_bwd(True, g, ref_m2, p)
    rdx2, rdb2 = oracle.bias_relu_dropout_bwd(g, ref_m2, p)
    assert_close(dx2, rdx2, "ragged brd bwd dx")
    assert_close(db2, rdb2, "ragged brd bwd dbias")


def test_in_place_and_no_mask_and_no_bias_grad():
    require_gpu()
    shape = (64, 512)
    x = synth.normal(5, "ip/x", shape, 0.0, 1.0, "f16")
    r = synth.normal(5, "ip/r", shape, 0.0, 1.0, "f16")
    b = synth.normal(5, "ip/b", (512,), 0.0, 0.02, "f16")
    ref, ref_mask = oracle.bias_dropout_residual_fwd(x, b, r, 0.1, 1, 2)
    xt = dev(x)
    ls_ops.ls_bias_dropout_residual_fwd(xt, None, xt, dev(b), dev(r), 0.1, 1, 2)  # out = x
    torch.cuda.synchronize()
    assert_close(f64(xt), ref, "in-place bdr fwd")
    rt = dev(r)
    ls_ops.ls_bias_dropout_residual_fwd(rt, None, dev(x), dev(b), rt, 0.1, 1, 2)  # out = residual
    torch.cuda.synchronize()
    assert_close(f64(rt), ref, "in-place (residual) bdr fwd")
    # dx written over dout, no bias gradient (and so no workspace)
    g = synth.normal(5, "ip/g", shape, 0.0, 1.0, "f16")
    gt = dev(g)
    ls_ops.ls_bias_dropout_residual_bwd(gt, None, gt, dev(ref_mask.view(np.int32)), 0.1)
    torch.cuda.synchronize()
    assert_close(f64(gt), oracle.bias_dropout_residual_bwd(g, ref_mask, 0.1)[0], "in-place bwd")


def test_empty_batch_zeroes_bias_grad():
    require_gpu()
    db = torch.full((64,), 7.0, dtype=torch.float16, device="cuda")
    empty = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    ls_ops.ls_bias_dropout_residual_bwd(empty, db, empty, None, 0.1)
    torch.cuda.synchronize()
    assert (db == 0).all()


def test_bias_grad_is_deterministic():
    require_gpu()
    L = synth.BERT_BASE
    d = synth.layer_inputs(L, 1, which={"ffn1_x", "ffn1_bias", "ffn1_dout"})
    _, m = oracle.bias_relu_dropout_fwd(d["ffn1_x"][:512], d["ffn1_bias"], 0.1, 0, 0)
    dout = d["ffn1_dout"][:512]
    a = run_dropout_bwd(True, dout, m, 0.1)
    b = run_dropout_bwd(True, dout, m, 0.1)
    np.testing.assert_array_equal(a[1], b[1])
    np.testing.assert_array_equal(a[0], b[0])

