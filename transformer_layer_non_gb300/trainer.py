"""Symbolic tensor linking for the fused trainer update ("LightSeq2",
section 2.3; "CMU 11-868 L10 (LightSeq)", technique 3, slide p.29).

At set-up, every parameter of a model is copied into one contiguous
workspace and re-pointed at its slice of it, and the same is done for the
gradients; the optimiser state (two FP32 moments) is one contiguous buffer
each.  The whole model then updates with a single ``ls_adam_update`` launch
instead of one launch per parameter tensor.  Only torch views are created:
writes through a parameter land in the workspace and the other way round.

Each slice starts on a 16-byte boundary (the kernel's vector accesses need
it); the few padding elements between slices are part of the update (their
parameters, gradients and moments stay zero, so they stay zero).
"""
from __future__ import annotations

from typing import Iterable, List

from . import ls_ops

ALIGN_BYTES = 16


class LinkedParameters:
    """One flat parameter workspace, one flat gradient workspace and the FP32
    Adam moments for a list of same-dtype parameter tensors (torch
    ``nn.Parameter`` or plain tensors with ``requires_grad``)."""

    def __init__(self, params: Iterable):
        import torch

        self.params: List = list(params)
        if not self.params:
            raise ValueError("no parameters to link")
        dtype, device = self.params[0].dtype, self.params[0].device
        for p in self.params:
            if p.dtype != dtype or p.device != device:
                raise ValueError("all linked parameters must share one dtype and device")
        esize = torch.empty((), dtype=dtype).element_size()
        step = ALIGN_BYTES // esize
        self.offsets = []
        n = 0
        for p in self.params:
            self.offsets.append(n)
            n += (p.numel() + step - 1) // step * step
        self.numel = n
        self.param_ws = torch.zeros(n, dtype=dtype, device=device)
        self.grad_ws = torch.zeros(n, dtype=dtype, device=device)
        self.exp_avg = torch.zeros(n, dtype=torch.float32, device=device)
        self.exp_avg_sq = torch.zeros(n, dtype=torch.float32, device=device)
        self.step = 0
        with torch.no_grad():
            for p, off in zip(self.params, self.offsets):
                k = p.numel()
                self.param_ws[off:off + k].copy_(p.detach().reshape(-1))
                p.data = self.param_ws[off:off + k].view(p.shape)
                if p.grad is not None:
                    self.grad_ws[off:off + k].copy_(p.grad.reshape(-1))
                p.grad = self.grad_ws[off:off + k].view(p.shape)

    def zero_grad(self):
        self.grad_ws.zero_()

    def adam_step(self, lr: float, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                  weight_decay: float = 0.0, grad_scale: float = 1.0, stream=None):
        """One fused Adam update of every linked parameter (one launch)."""
        self.step += 1
        ls_ops.ls_adam_update(self.param_ws, self.grad_ws, self.exp_avg, self.exp_avg_sq, lr,
                              beta1, beta2, eps, weight_decay, self.step, grad_scale,
                              stream=stream)
