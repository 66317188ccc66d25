"""GPU parity at the largest index ranges the dropout kernels handle.

A bias+ReLU+dropout forward over 2^34 + 2^20 FP16 elements (4096 columns):
more than 2^31 16-byte vectors, so the forward takes its 64-bit index path,
and Philox counter blocks (element index / 4) past 2^32, so the counter's
second word is nonzero for the last 2^20 elements.  The offset has its high
word set too.  The oracle cannot redo 17 G elements in seconds, so sampled
elements (random ones, the first and last ones, and the ones around the
counter-block boundary) are checked one by one against the oracle's Philox
words: the mask bit exactly, the value within |err| <= 2e-3 + 2e-3*|ref|.
Then the bias+dropout+residual backward without a saved mask (keep bits
redrawn from seed and offset) runs over the same range and is checked the
same way.  About 72 GB of device memory; skipped on smaller devices."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import require_gpu
from transformer_layer_non_gb300 import ls_ops

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

COLS = 4096
N = (1 << 34) + (1 << 20)
ROWS = N // COLS
P = 0.1
SEED = 0x0123456789ABCDEF
OFFSET = (7 << 32) | 5
PAD = 4096  # guard bytes on each side of an output


def _guarded(nbytes):
    """A byte buffer with canary-filled guard bands; returns (buffer, body)."""
    buf = torch.empty(nbytes + 2 * PAD, dtype=torch.uint8, device="cuda")
    buf[:PAD].fill_(0xA5)
    buf[-PAD:].fill_(0xA5)
    return buf, buf[PAD:PAD + nbytes]


def _guards_intact(buf):
    return bool((buf[:PAD] == 0xA5).all()) and bool((buf[-PAD:] == 0xA5).all())


def _samples():
    rng = np.random.default_rng(20)
    idx = np.concatenate([
        rng.integers(0, N, 4000, dtype=np.int64),
        np.arange(0, 64), np.arange(N - 64, N),
        (1 << 34) + np.arange(-64, 64),                # counter block 2^32 boundary
        (1 << 34) + rng.integers(0, 1 << 20, 500),     # blocks with a nonzero second word
    ]).astype(np.int64)
    return np.unique(idx)


def _tol_ok(got, ref):
    return np.abs(got - ref) <= 2e-3 + 2e-3 * np.abs(ref)


def test_dropout_past_32_bit_indices():
    require_gpu()
    free, _ = torch.cuda.mem_get_info()
    need = 2 * N * 2 + N // 8 + (1 << 30)
    if free < need:
        pytest.skip(f"needs {need / 1e9:.0f} GB of free device memory, {free / 1e9:.0f} GB free")
    g = torch.Generator(device="cuda").manual_seed(1)
    xbuf, xb = _guarded(N * 2)
    x = xb.view(torch.float16).view(ROWS, COLS)
    x.normal_(0.0, 1.0, generator=g)
    bias = (torch.randn(COLS, generator=g, device="cuda") * 0.02).half()
    obuf, ob = _guarded(N * 2)
    out = ob.view(torch.float16).view(ROWS, COLS)
    mbuf, mb = _guarded(N // 8)
    mask = mb.view(torch.int32)

    ls_ops.ls_bias_relu_dropout_fwd(out, mask, x, bias, P, SEED, OFFSET)
    torch.cuda.synchronize()
    assert _guards_intact(obuf) and _guards_intact(mbuf)
    assert ls_ops.check_device_errors() == 0

    idx = _samples()
    it = torch.from_numpy(idx).cuda()
    xs = x.view(-1)[it].double().cpu().numpy()
    os_ = out.view(-1)[it].double().cpu().numpy()
    words = mask.view(-1)[torch.from_numpy(idx >> 5).cuda()].cpu().numpy().view(np.uint32)
    bits = (words >> (idx & 31).astype(np.uint32)) & 1
    bs = bias.double().cpu().numpy()[idx % COLS]
    thr = oracle.dropout_threshold(P)
    scale = 1.0 / (1.0 - np.float32(P))
    keep = np.array([oracle.dropout_word(SEED, OFFSET, int(i)) >= thr for i in idx])
    z = xs + bs
    on = keep & (z > 0)
    np.testing.assert_array_equal(bits.astype(bool), on, "ReLU-and-keep bits")
    ref = np.where(on, z * scale, 0.0)
    assert _tol_ok(os_, ref).all(), f"forward: max err {np.abs(os_ - ref).max()}"
    kept = keep.mean()
    assert abs(kept - (1 - P)) < 0.03, kept

    # Backward with the keep bits redrawn from (seed, offset): dout = the
    # forward output, dx written over x (exact aliasing is not used here).
    del mask, mbuf, mb
    ls_ops.ls_bias_dropout_residual_bwd(x, None, out, None, P, SEED, OFFSET)
    torch.cuda.synchronize()
    assert _guards_intact(xbuf)
    assert ls_ops.check_device_errors() == 0
    dx = x.view(-1)[it].double().cpu().numpy()
    ref_dx = np.where(keep, os_ * scale, 0.0)
    assert _tol_ok(dx, ref_dx).all(), f"backward: max err {np.abs(dx - ref_dx).max()}"
