"""GPU parity: LayerNorm forward (single-sync statistics) and backward (two-sum
form with fused gamma/beta gradients) against the FP64 oracle, every element,
|err| <= 2e-3 + 2e-3*|ref|.  Widths cover every row-length class of the
dispatch (lanes per row 1..32, 1..8 vectors per lane, CTA per row)."""
import numpy as np
import pytest

import oracle
from transformer_layer_non_gb300 import ls_ops, synth
from tests.gpu_util import Guarded, assert_close, dev, f64, require_gpu, tdtype

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EPS = 1e-5


def run_fwd(x, g, b, eps=EPS, in_place=False):
    rows, cols = x.shape
    mean = Guarded((rows,), torch.float32)
    rstd = Guarded((rows,), torch.float32)
    if in_place:
        xt = dev(x)
        ls_ops.ls_layernorm_fwd(xt, mean.t, rstd.t, xt, dev(g), dev(b), eps)
        torch.cuda.synchronize()
        y = xt
    else:
        yg = Guarded(x.shape, tdtype(x.dtype))
        ls_ops.ls_layernorm_fwd(yg.t, mean.t, rstd.t, dev(x), dev(g), dev(b), eps)
        torch.cuda.synchronize()
        yg.check()
        y = yg.t
    mean.check()
    rstd.check()
    return f64(y), mean.t.cpu().numpy(), rstd.t.cpu().numpy()


def run_bwd(dy, x, g, mean32, rstd32):
    rows, cols = x.shape
    dx = Guarded(x.shape, tdtype(x.dtype))
    dg = Guarded((cols,), tdtype(x.dtype))
    db = Guarded((cols,), tdtype(x.dtype))
    ws = torch.empty(max(ls_ops.colreduce_workspace_bytes(rows, cols), 16), dtype=torch.uint8,
                     device="cuda").fill_(0xFF)  # garbage: the workspace needs no init
    ls_ops.ls_layernorm_bwd(dx.t, dg.t, db.t, dev(dy), dev(x), dev(g), dev(mean32), dev(rstd32),
                            workspace=ws)
    torch.cuda.synchronize()
    for t in (dx, dg, db):
        t.check()
    return f64(dx.t), f64(dg.t), f64(db.t)


def check_case(x, g, b, dy, what):
    y, mean, rstd = run_fwd(x, g, b)
    ry, rmean, rrstd = oracle.layernorm_fwd(x, g, b, EPS)
    assert_close(y, ry, f"{what} y")
    np.testing.assert_allclose(mean, rmean, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(rstd, rrstd, rtol=1e-4)
    rdx, rdg, rdb = oracle.layernorm_bwd(dy, x, g, EPS)
    # (a) the backward fed the oracle's statistics, rounded to FP32
    dx, dg, db = run_bwd(dy, x, g, rmean.astype(np.float32), rrstd.astype(np.float32))
    assert_close(dx, rdx, f"{what} dx")
    assert_close(dg, rdg, f"{what} dgamma")
    assert_close(db, rdb, f"{what} dbeta")
    # (b) chained: the backward fed the GPU forward's own statistics
    dx2, dg2, db2 = run_bwd(dy, x, g, mean, rstd)
    assert_close(dx2, rdx, f"{what} chained dx")
    assert_close(dg2, rdg, f"{what} chained dgamma")
    assert_close(db2, rdb, f"{what} chained dbeta")


@pytest.mark.parametrize("name", ["tiny", "transformer-base", "bert-base", "gpt2-large"])
def test_layer_configs(name):
    require_gpu()
    L = synth.LAYERS[name]
    d = synth.layer_inputs(L, 0, which={"ln1_x", "ln1_dy", "ln1_gamma", "ln1_beta"})
    check_case(d["ln1_x"], d["ln1_gamma"], d["ln1_beta"], d["ln1_dy"], name)


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("cols", [8, 16, 24, 64, 136, 256, 264, 512, 768, 1280, 2048, 2056,
                                  4096, 8192, 16384])
def test_widths(dtype, cols):
    require_gpu()
    rows = 37 if cols <= 4096 else 5
    shape = (rows, cols)
    x = synth.normal(1, f"lnw/x{cols}", shape, 0.0, 1.0, dtype)
    g = synth.normal(1, f"lnw/g{cols}", (cols,), 1.0, 0.1, dtype)
    b = synth.normal(1, f"lnw/b{cols}", (cols,), 0.0, 0.1, dtype)
    dy = synth.normal(1, f"lnw/dy{cols}", shape, 0.0, 1.0, dtype)
    check_case(x, g, b, dy, f"{dtype} H={cols}")


def test_many_rows_per_cta_and_ragged_rows():
    # 10007 rows: several row steps per backward CTA and a ragged last CTA.
    require_gpu()
    shape = (10007, 520)
    x = synth.normal(2, "lnr/x", shape, 0.0, 1.0, "f16")
    g = synth.normal(2, "lnr/g", (520,), 1.0, 0.1, "f16")
    b = synth.normal(2, "lnr/b", (520,), 0.0, 0.1, "f16")
    dy = synth.normal(2, "lnr/dy", shape, 0.0, 1.0, "f16")
    check_case(x, g, b, dy, "10007x520")


@pytest.mark.parametrize("cols", [1024, 1280, 1536, 1792, 2048])
def test_wide_rows_two_buffers(cols):
    # FP16 rows of 4..8 vectors per lane keep two row buffers in the forward
    # (the second row's loads in flight, x - K formed again in the output
    # pass); 9001 rows give every warp 2-4 rows, so both buffers are used more
    # than once, and a ragged last round.
    require_gpu()
    shape = (9001, cols)
    x = synth.normal(3, f"lnd/x{cols}", shape, 0.5, 2.0, "f16")
    g = synth.normal(3, f"lnd/g{cols}", (cols,), 1.0, 0.1, "f16")
    b = synth.normal(3, f"lnd/b{cols}", (cols,), 0.0, 0.1, "f16")
    dy = synth.normal(3, f"lnd/dy{cols}", shape, 0.0, 1.0, "f16")
    check_case(x, g, b, dy, f"9001x{cols}")


def test_large_mean_rows_fp32():
    # Rows with mean 1e4 and unit spread: a naive one-pass variance in FP32
    # loses every digit here; the sums about the first element do not.
    require_gpu()
    shape = (16, 512)
    x = (synth.normal(4, "lnm/x", shape, 0.0, 1.0, "f32").astype(np.float64) + 1e4).astype(
        np.float32)
    g = np.ones(512, np.float32)
    b = np.zeros(512, np.float32)
    y, mean, rstd = run_fwd(x, g, b)
    ry, rmean, rrstd = oracle.layernorm_fwd(x, g, b, EPS)
    assert_close(y, ry, "large-mean y")
    np.testing.assert_allclose(rstd, rrstd, rtol=1e-3)


def test_in_place_and_no_stats_and_no_param_grads():
    require_gpu()
    shape = (64, 768)
    x = synth.normal(6, "lni/x", shape, 0.0, 1.0, "f16")
    g = synth.normal(6, "lni/g", (768,), 1.0, 0.1, "f16")
    b = synth.normal(6, "lni/b", (768,), 0.0, 0.1, "f16")
    y, _, _ = run_fwd(x, g, b, in_place=True)
    ry, rmean, rrstd = oracle.layernorm_fwd(x, g, b, EPS)
    assert_close(y, ry, "in-place y")
    # mean/rstd are optional outputs
    yt = torch.empty(shape, dtype=torch.float16, device="cuda")
    ls_ops.ls_layernorm_fwd(yt, None, None, dev(x), dev(g), dev(b), EPS)
    torch.cuda.synchronize()
    assert_close(f64(yt), ry, "no-stats y")
    # backward with dx over dy, without dgamma/dbeta (no workspace)
    dy = synth.normal(6, "lni/dy", shape, 0.0, 1.0, "f16")
    dyt = dev(dy)
    ls_ops.ls_layernorm_bwd(dyt, None, None, dyt, dev(x), dev(g), dev(rmean.astype(np.float32)),
                            dev(rrstd.astype(np.float32)))
    torch.cuda.synchronize()
    assert_close(f64(dyt), oracle.layernorm_bwd(dy, x, g, EPS)[0], "in-place dx")


def test_param_grads_deterministic_and_empty_batch():
    require_gpu()
    L = synth.GPT2_LARGE
    d = synth.layer_inputs(L, 3, which={"ln2_x", "ln2_dy", "ln2_gamma"})
    x, dy, g = d["ln2_x"], d["ln2_dy"], d["ln2_gamma"]
    _, m, r = oracle.layernorm_fwd(x, g, np.zeros_like(g), EPS)
    a = run_bwd(dy, x, g, m.astype(np.float32), r.astype(np.float32))
    c = run_bwd(dy, x, g, m.astype(np.float32), r.astype(np.float32))
    for u, v in zip(a, c):
        np.testing.assert_array_equal(u, v)
    dg = torch.full((1280,), 3.0, dtype=torch.float16, device="cuda")
    db = torch.full((1280,), 3.0, dtype=torch.float16, device="cuda")
    e = torch.empty((0, 1280), dtype=torch.float16, device="cuda")
    ls_ops.ls_layernorm_bwd(e, dg, db, e, e, dev(g), None, None)
    torch.cuda.synchronize()
    assert (dg == 0).all() and (db == 0).all()
