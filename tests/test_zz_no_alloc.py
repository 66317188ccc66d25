"""ls_layernorm_bwd_noalloc: the LayerNorm backward for callers that cannot
allocate device memory (a plugin inside a host application that owns every
device allocation, or code where cudaMalloc may not be called) and so cannot
pass the workspace for the gamma/beta partial sums.  Those sums live in a
scratch array built into the library instead.

Checked through the C ABI on two calls in a row (the second finds the first
call's leftovers in the shared scratch): dx, dgamma and dbeta bit for bit equal
to ls_layernorm_bwd with a caller workspace (the same kernels and fixed-order
reductions), and within the parity tolerance of the FP64 oracle.  A shape whose
partial sums do not fit is rejected on real buffers, which stay untouched.  In
a second CUDA context on the same device (a child process) the entry point
uses that context's own copy of the array.  This file is collected last and
also passes when run on its own."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from transformer_layer_non_gb300 import ls_ops, synth
from tests.gpu_util import assert_close, dev, f64, require_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EPS = 1e-5
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(seed, rows, cols):
    x = synth.normal(seed, f"na/x{cols}", (rows, cols), 0.0, 1.0, "f16")
    dy = synth.normal(seed, f"na/dy{cols}", (rows, cols), 0.0, 1.0, "f16")
    g = synth.normal(seed, f"na/g{cols}", (cols,), 1.0, 0.1, "f16")
    _, mean, rstd = oracle.layernorm_fwd(x, g, np.zeros_like(g), EPS)
    return x, dy, g, mean.astype(np.float32), rstd.astype(np.float32)


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


def _bits(t):
    return t.cpu().view(torch.int16).numpy()


def test_no_alloc_matches_workspace_entry_point_bitwise_on_two_calls():
    require_gpu()
    # GPT-2-large width, then BERT-base width: the second call reuses the
    # scratch the first one left behind.
    for seed, rows, cols in [(1, 4096, 1280), (2, 4096, 768)]:
        host = _inputs(seed, rows, cols)
        args = [dev(a) for a in host]
        got = _no_alloc(*args)
        ref = _with_workspace(*args)
        torch.cuda.synchronize()
        for name, a, b in zip(("dx", "dgamma", "dbeta"), got, ref):
            np.testing.assert_array_equal(_bits(a), _bits(b),
                                          f"no-alloc {name} ({rows}x{cols}) differs in bits")
        rdx, rdg, rdb = oracle.layernorm_bwd(host[1], host[0], host[2], EPS)
        for name, a, r in zip(("dx", "dgamma", "dbeta"), got, (rdx, rdg, rdb)):
            assert_close(f64(a), r, f"no-alloc {name} ({rows}x{cols}) vs oracle")


def test_no_alloc_rejects_shapes_beyond_its_scratch():
    require_gpu()
    cols = 16384
    # The fewest rows whose partial sums exceed the scratch (real, small buffers).
    rows = next(r for r in range(1, 4097)
                if ls_ops.colreduce_workspace_bytes(r, cols) > ls_ops.LS_NOALLOC_SCRATCH_BYTES)
    x, dy, g, mean, rstd = (dev(a) for a in _inputs(3, rows, cols))
    dx, dg, db = torch.empty_like(x), torch.empty_like(g), torch.empty_like(g)
    for t in (dx, dg, db):
        t.view(torch.uint8).fill_(0x5A)
    st = ls_ops.load().ls_layernorm_bwd_noalloc(
        ls_ops.LS_F16, dx.data_ptr(), dg.data_ptr(), db.data_ptr(), dy.data_ptr(), x.data_ptr(),
        g.data_ptr(), mean.data_ptr(), rstd.data_ptr(), rows, cols, None)
    torch.cuda.synchronize()
    assert st == ls_ops.LS_ERR_UNSUPPORTED_SHAPE, ls_ops.status_string(st)
    assert "scratch" in ls_ops.last_error()
    for t in (dx, dg, db):
        assert bool((t.view(torch.uint8) == 0x5A).all()), "a rejected call wrote an output"


# A child process: the entry point in the primary context, then in a second
# context created with the driver API on the same device (its own buffers),
# then in the primary context again; all three results must be the same bits.
_CHILD = r"""
import ctypes, sys
import numpy as np
sys.path.insert(0, ROOT)
import torch
import oracle
from transformer_layer_non_gb300 import ls_ops, synth

rows, cols, eps = 512, 768, 1e-5
x = synth.normal(4, "na/ctx/x", (rows, cols), 0.0, 1.0, "f16")
dy = synth.normal(4, "na/ctx/dy", (rows, cols), 0.0, 1.0, "f16")
g = synth.normal(4, "na/ctx/g", (cols,), 1.0, 0.1, "f16")
_, mean, rstd = oracle.layernorm_fwd(x, g, np.zeros_like(g), eps)
mean, rstd = mean.astype(np.float32), rstd.astype(np.float32)
host_in = [x, dy, g, mean, rstd]

def primary():
    t = [torch.from_numpy(a).cuda() for a in host_in]
    dx, dg, db = torch.empty_like(t[0]), torch.empty_like(t[2]), torch.empty_like(t[2])
    ls_ops.ls_layernorm_bwd_noalloc(dx, dg, db, t[1], t[0], t[2], t[3], t[4])
    torch.cuda.synchronize()
    return [a.cpu().numpy() for a in (dx, dg, db)]

lib = ls_ops.load(build_if_needed=False)
r1 = primary()

cu = ctypes.CDLL("libcuda.so.1")
def ck(r, what):
    if r != 0:
        raise SystemExit(f"{what}: CUresult {r}")
P = ctypes.c_void_p
ctx = P()
if hasattr(cu, "cuCtxCreate_v2"):
    ck(cu.cuCtxCreate_v2(ctypes.byref(ctx), ctypes.c_uint(0), ctypes.c_int(0)), "cuCtxCreate")
else:
    ck(cu.cuCtxCreate_v4(ctypes.byref(ctx), None, ctypes.c_uint(0), ctypes.c_int(0)), "cuCtxCreate")
cu.cuMemAlloc_v2.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_size_t]
cu.cuMemcpyHtoD_v2.argtypes = [ctypes.c_uint64, P, ctypes.c_size_t]
cu.cuMemcpyDtoH_v2.argtypes = [P, ctypes.c_uint64, ctypes.c_size_t]
cu.cuMemFree_v2.argtypes = [ctypes.c_uint64]
def alloc(nbytes):
    p = ctypes.c_uint64()
    ck(cu.cuMemAlloc_v2(ctypes.byref(p), nbytes), "cuMemAlloc")
    return p.value
ins = []
for a in host_in:
    a = np.ascontiguousarray(a)
    p = alloc(a.nbytes)
    ck(cu.cuMemcpyHtoD_v2(p, a.ctypes.data, a.nbytes), "cuMemcpyHtoD")
    ins.append(p)
outs = [np.empty_like(x), np.empty_like(g), np.empty_like(g)]
dptr = [alloc(o.nbytes) for o in outs]
st = lib.ls_layernorm_bwd_noalloc(ls_ops.LS_F16, dptr[0], dptr[1], dptr[2], ins[1], ins[0],
                                  ins[2], ins[3], ins[4], rows, cols, None)
if st != 0:
    raise SystemExit("second context: " + ls_ops.status_string(st) + " " + ls_ops.last_error())
ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
for o, p in zip(outs, dptr):
    ck(cu.cuMemcpyDtoH_v2(o.ctypes.data, p, o.nbytes), "cuMemcpyDtoH")
for p in ins + dptr:
    ck(cu.cuMemFree_v2(p), "cuMemFree")
old = P()
ck(cu.cuCtxPopCurrent_v2(ctypes.byref(old)), "cuCtxPopCurrent")
r2 = outs
r3 = primary()
ck(cu.cuCtxDestroy_v2(ctx), "cuCtxDestroy")
for name, a, b, c in zip(("dx", "dgamma", "dbeta"), r1, r2, r3):
    if not (np.array_equal(a.view(np.int16), b.view(np.int16))
            and np.array_equal(a.view(np.int16), c.view(np.int16))):
        raise SystemExit(f"{name}: results differ between contexts")
print("contexts agree")
"""


def test_no_alloc_in_a_second_context_on_the_same_device():
    require_gpu()
    code = "ROOT = " + repr(ROOT) + "\n" + _CHILD
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "contexts agree" in r.stdout, r.stdout + r.stderr
