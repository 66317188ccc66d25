"""Symbolic tensor linking (host-side logic, on CPU): every parameter becomes
a view of one contiguous workspace at a 16-byte-aligned offset, its gradient
a view of the gradient workspace; values survive the move, writes through
either side are shared, and padding stays zero.  The GPU test runs one fused
update over linked parameters against torch.optim.AdamW."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from transformer_layer_non_gb300.trainer import LinkedParameters  # noqa: E402


def _params(dtype=torch.float16, device="cpu"):
    g = torch.Generator().manual_seed(0)
    shapes = [(3, 5), (7,), (2, 2, 3), (1,), (16,)]
    ps = []
    for s in shapes:
        p = torch.nn.Parameter(torch.randn(*s, generator=g).to(dtype).to(device))
        p.grad = torch.randn(*s, generator=g).to(dtype).to(device)
        ps.append(p)
    return ps


def test_views_offsets_and_sharing():
    ps = _params()
    before = [p.detach().clone() for p in ps]
    grads = [p.grad.clone() for p in ps]
    lp = LinkedParameters(ps)
    for p, off, b, gr in zip(ps, lp.offsets, before, grads):
        assert off % 8 == 0  # 16 bytes of FP16
        assert p.data.data_ptr() == lp.param_ws.data_ptr() + off * 2
        assert p.grad.data_ptr() == lp.grad_ws.data_ptr() + off * 2
        assert torch.equal(p.detach(), b) and torch.equal(p.grad, gr)
    assert lp.numel == sum((p.numel() + 7) // 8 * 8 for p in ps)
    used = torch.zeros(lp.numel, dtype=torch.bool)
    for p, off in zip(ps, lp.offsets):
        used[off:off + p.numel()] = True
    assert not lp.param_ws[~used].any() and not lp.grad_ws[~used].any()
    with torch.no_grad():
        ps[1].add_(1.0)
    assert torch.equal(lp.param_ws[lp.offsets[1]:lp.offsets[1] + 7], ps[1].detach())
    lp.zero_grad()
    assert all(not p.grad.any() for p in ps)


def test_rejects_mixed_dtypes():
    ps = _params()
    ps.append(torch.nn.Parameter(torch.zeros(4)))
    with pytest.raises(ValueError):
        LinkedParameters(ps)


@pytest.mark.gpu
def test_linked_update_matches_adamw_on_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ps = _params(torch.float32, "cuda")
    ref = [torch.nn.Parameter(p.detach().clone()) for p in ps]
    for r, p in zip(ref, ps):
        r.grad = p.grad.clone()
    lp = LinkedParameters(ps)
    opt = torch.optim.AdamW(ref, lr=1e-2, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    for _ in range(3):
        lp.adam_step(1e-2, weight_decay=0.01)
        opt.step()
    torch.cuda.synchronize()
    for p, r in zip(ps, ref):
        np.testing.assert_allclose(p.detach().cpu().numpy(), r.detach().cpu().numpy(),
                                   rtol=1e-5, atol=1e-6)
