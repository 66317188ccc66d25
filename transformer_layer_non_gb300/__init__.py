"""Fused non-GEMM Transformer-layer operators for GB300 (sm_103a).

The operators -- bias+dropout+residual, bias+ReLU+dropout, LayerNorm and
masked attention softmax, forward and backward -- live in the C-ABI library
``libls_ops.so`` (declared in ``include/ls_ops.h``); :mod:`.ls_ops` binds it.
"""
from . import ls_ops  # noqa: F401

__all__ = ["ls_ops"]
