"""Failure detection on the GPU without a fault: the library's bounded wait
runs out on a barrier that nothing completes (the self-test entry point), the
kernel records LS_DEVERR_WAIT_TIMEOUT and returns, ls_check_device_errors
reports the flag once and clears it, and the context stays usable (an
ordinary operator afterwards still matches the oracle)."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_close, dev, f64, require_gpu
from transformer_layer_non_gb300 import ls_ops, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared():
    require_gpu()
    assert ls_ops.check_device_errors() == 0  # nothing pending from earlier work
    ls_ops.selftest_wait_timeout(polls=256)
    assert ls_ops.check_device_errors() == ls_ops.LS_DEVERR_WAIT_TIMEOUT
    assert ls_ops.check_device_errors() == 0  # read once, then cleared
    # The context is healthy: a softmax afterwards still matches the oracle.
    x, dy, kl = synth.sweep_inputs(512, seed=4, elements=1 << 14)
    y = torch.empty(x.shape, dtype=torch.float16, device="cuda")
    ls_ops.ls_softmax_fwd(y, dev(x), dev(kl), False)
    torch.cuda.synchronize()
    assert_close(f64(y), oracle.softmax_fwd(x, kl, False), "softmax after the self-test")
    assert ls_ops.check_device_errors() == 0


def test_selftest_argument_check():
    require_gpu()
    with pytest.raises(ls_ops.LsError):
        ls_ops.selftest_wait_timeout(polls=0)
