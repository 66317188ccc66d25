"""Column reductions forked onto a second stream (ls_set_reduction_stream /
ls_join_reductions) give the same bits as the default schedule: dx and the
bias, gamma and beta gradients of every backward entry with a column
reduction, eagerly and inside a captured CUDA graph; with one shared
workspace (the library orders the later call after the pending reduction);
and past the 16 pending reductions the library tracks.  The default results
themselves are checked against the oracle by the per-operator tests."""
import numpy as np
import pytest

from tests.gpu_util import dev, require_gpu
from transformer_layer_non_gb300 import ls_ops

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

T, H, F = 4096, 768, 3072
P = 0.1


def _inputs():
    g = np.random.default_rng(5)
    t = {
        "ln_x": g.normal(0, 1, (T, H)).astype(np.float16),
        "ln_dy": g.normal(0, 1, (T, H)).astype(np.float16),
        "gamma": g.normal(1, 0.1, H).astype(np.float16),
        "beta": g.normal(0, 0.1, H).astype(np.float16),
        "bdr_dout": g.normal(0, 1, (T, H)).astype(np.float16),
        "brd_x": g.normal(0, 1, (T, F)).astype(np.float16),
        "brd_bias": g.normal(0, 0.1, F).astype(np.float16),
        "brd_dout": g.normal(0, 1, (T, F)).astype(np.float16),
        "qkv": g.normal(0, 1, (3, 8, 12, 512, 64)).astype(np.float16),
    }
    d = {k: dev(v) for k, v in t.items()}
    e = lambda *s, dt=torch.float16: torch.empty(s, dtype=dt, device="cuda")  # noqa: E731
    d["mean"], d["rstd"] = e(T, dt=torch.float32), e(T, dt=torch.float32)
    ls_ops.ls_layernorm_fwd(e(T, H), d["mean"], d["rstd"], d["ln_x"], d["gamma"], d["beta"])
    d["bdr_mask"] = e((T * H + 31) // 32, dt=torch.int32)
    ls_ops.ls_bias_dropout_residual_fwd(e(T, H), d["bdr_mask"], d["ln_x"], d["gamma"],
                                        d["ln_dy"], P, 7, 0)
    d["brd_mask"] = e((T * F + 31) // 32, dt=torch.int32)
    ls_ops.ls_bias_relu_dropout_fwd(e(T, F), d["brd_mask"], d["brd_x"], d["brd_bias"], P, 7, 1)
    torch.cuda.synchronize()
    return d


def _outputs():
    e = lambda *s: torch.full(s, float("nan"), dtype=torch.float16, device="cuda")  # noqa: E731
    return {"ln_dx": e(T, H), "dgamma": e(H), "dbeta": e(H), "bdr_dx": e(T, H),
            "bdr_dbias": e(H), "brd_dx": e(T, F), "brd_dbias": e(F), "dqkv": e(T, 3 * H),
            "qkv_dbias": e(3 * H)}


def _calls(d, o, ws):
    """The four backward entries with a column reduction; ws: four workspaces
    (or one, four times)."""
    return [
        lambda: ls_ops.ls_layernorm_bwd(o["ln_dx"], o["dgamma"], o["dbeta"], d["ln_dy"],
                                        d["ln_x"], d["gamma"], d["mean"], d["rstd"],
                                        workspace=ws[0]),
        lambda: ls_ops.ls_bias_dropout_residual_bwd(o["bdr_dx"], o["bdr_dbias"], d["bdr_dout"],
                                                    d["bdr_mask"], P, workspace=ws[1]),
        lambda: ls_ops.ls_bias_relu_dropout_bwd(o["brd_dx"], o["brd_dbias"], d["brd_dout"],
                                                d["brd_mask"], P, workspace=ws[2]),
        lambda: ls_ops.ls_bias_reshape_qkv_bwd(o["dqkv"], o["qkv_dbias"], d["qkv"], 8, 512, 12,
                                               workspace=ws[3]),
    ]


def _workspaces(n):
    return [ls_ops.new_workspace([(T, F), (T, 3 * H)]) for _ in range(n)]


def _bits(o):
    return {k: v.view(torch.int16).cpu().numpy() for k, v in o.items()}


def _same(a, b, what):
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], f"{what}: {k}")


@pytest.fixture(scope="module")
def ref():
    require_gpu()
    d = _inputs()
    o = _outputs()
    ws = _workspaces(1) * 4
    for fn in _calls(d, o, ws):
        fn()
    torch.cuda.synchronize()
    return d, _bits(o)


def _run_forked(d, ws, side, main=None):
    o = _outputs()
    main = main or torch.cuda.current_stream()
    ls_ops.set_reduction_stream(side)
    try:
        with torch.cuda.stream(main):
            for fn in _calls(d, o, ws):
                fn()
            ls_ops.join_reductions()
    finally:
        ls_ops.set_reduction_stream(None)
    torch.cuda.synchronize()
    return _bits(o)


def test_forked_reductions_same_bits(ref):
    d, want = ref
    side = torch.cuda.Stream()
    _same(want, _run_forked(d, _workspaces(4), side), "own workspaces")


def test_shared_workspace_is_ordered(ref):
    d, want = ref
    side = torch.cuda.Stream()
    _same(want, _run_forked(d, _workspaces(1) * 4, side), "one shared workspace")


def test_forked_reductions_in_a_graph(ref):
    d, want = ref
    side = torch.cuda.Stream()
    ws = _workspaces(4)
    o = _outputs()
    calls = _calls(d, o, ws)
    main = torch.cuda.Stream()
    main.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    ls_ops.set_reduction_stream(side)
    try:
        with torch.cuda.graph(g, stream=main):
            for fn in calls:
                fn()
            ls_ops.join_reductions()
    finally:
        ls_ops.set_reduction_stream(None)
    for v in o.values():
        v.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    _same(want, _bits(o), "graph replay")


def test_more_pending_than_tracked(ref):
    # 20 forks without a join: the library orders the main stream after the
    # oldest pending reduction when its table of 16 is full.
    d, want = ref
    side = torch.cuda.Stream()
    ws = _workspaces(20)
    o = _outputs()
    ls_ops.set_reduction_stream(side)
    try:
        for i in range(20):
            ls_ops.ls_bias_dropout_residual_bwd(o["bdr_dx"], o["bdr_dbias"], d["bdr_dout"],
                                                d["bdr_mask"], P, workspace=ws[i])
        ls_ops.join_reductions()
    finally:
        ls_ops.set_reduction_stream(None)
    torch.cuda.synchronize()
    got = _bits(o)
    np.testing.assert_array_equal(got["bdr_dbias"], want["bdr_dbias"])
    np.testing.assert_array_equal(got["bdr_dx"], want["bdr_dx"])


def test_reset_while_pending_is_refused(ref):
    d, _ = ref
    side = torch.cuda.Stream()
    o = _outputs()
    ws = _workspaces(1)
    ls_ops.set_reduction_stream(side)
    try:
        _calls(d, o, ws * 4)[1]()
        with pytest.raises(ls_ops.LsError) as ei:
            ls_ops.set_reduction_stream(None)
        assert ei.value.status == ls_ops.LS_ERR_INVALID_ARGUMENT
        ls_ops.join_reductions()
    finally:
        ls_ops.set_reduction_stream(None)
    torch.cuda.synchronize()


def test_noalloc_entry_follows_the_reduction_stream(ref):
    # The allocation-free LayerNorm backward forks like ls_layernorm_bwd; its
    # one built-in scratch is tracked as the pending reduction's workspace, so
    # a second call right after the first waits for the first reduction.
    d, want = ref
    side = torch.cuda.Stream()
    outs = [_outputs(), _outputs()]
    ls_ops.set_reduction_stream(side)
    try:
        for o in outs:
            ls_ops.ls_layernorm_bwd_noalloc(o["ln_dx"], o["dgamma"], o["dbeta"], d["ln_dy"],
                                            d["ln_x"], d["gamma"], d["mean"], d["rstd"])
        ls_ops.join_reductions()
    finally:
        ls_ops.set_reduction_stream(None)
    torch.cuda.synchronize()
    for o in outs:
        got = _bits(o)
        for k in ("ln_dx", "dgamma", "dbeta"):
            np.testing.assert_array_equal(got[k], want[k], k)
