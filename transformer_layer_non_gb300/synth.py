"""Seeded synthetic inputs shaped like the Transformer / BERT / GPT-2 layers.

This module only draws random numbers (numpy ``default_rng``) and rounds them
to the storage dtype; it holds none of the operators' arithmetic.  Tests feed
the same arrays to the CUDA library and to the CPU oracle; the benchmark uses
them as its device-resident inputs.

Distributions (one per tensor role): activations and upstream gradients
N(0, 1); gamma N(1, 0.1); beta N(0, 0.1); biases N(0, 0.02); attention scores
N(0, 3) (standard deviation 3).  Key-padding lengths are integers uniform on
[lo, seq]; the softmax sweep draws one length per row, uniform on [1, k_len].
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Layer:
    """One Transformer layer's non-GEMM workload."""
    name: str
    batch: int
    seq: int
    hidden: int
    heads: int
    ffn: int
    dtype: str                  # "f16" or "f32" storage
    pad_lo: Optional[int]       # key lengths ~ U[pad_lo, seq]; None: no padding mask
    causal: bool
    p: float = 0.1

    @property
    def tokens(self) -> int:
        return self.batch * self.seq


# The five workloads: four layers and the softmax sweep.
TINY = Layer("tiny", 2, 16, 64, 4, 256, "f32", None, False)
TRANSFORMER_BASE = Layer("transformer-base", 64, 64, 512, 8, 2048, "f16", 8, False)
BERT_BASE = Layer("bert-base", 8, 512, 768, 12, 3072, "f16", 128, False)
GPT2_LARGE = Layer("gpt2-large", 4, 1024, 1280, 20, 5120, "f16", None, True)
LAYERS: Dict[str, Layer] = {l.name: l for l in (TINY, TRANSFORMER_BASE, BERT_BASE, GPT2_LARGE)}

SWEEP_K_LENS = (16, 32, 64, 128, 256, 512, 1024, 2048, 4096)
SWEEP_ELEMENTS = 1 << 22


def np_dtype(dtype: str):
    return {"f16": np.float16, "f32": np.float32}[dtype]


def _rng(seed: int, role: str) -> np.random.Generator:
    # A distinct, stable stream per (seed, tensor role).
    return np.random.default_rng([seed, zlib.crc32(role.encode())])


def normal(seed: int, role: str, shape, mean: float, std: float, dtype: str) -> np.ndarray:
    """N(mean, std) drawn in float64, rounded once to the storage dtype."""
    a = _rng(seed, role).standard_normal(shape)
    if std != 1.0:
        a *= std
    if mean != 0.0:
        a += mean
    return a.astype(np_dtype(dtype))


def key_lengths(seed: int, role: str, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform on [lo, hi] (inclusive), int32."""
    return _rng(seed, role).integers(lo, hi + 1, size=n).astype(np.int32)


def layer_inputs(layer: Layer, seed: int = 0, which=None) -> Dict[str, np.ndarray]:
    """Inputs of every operator of one layer, forward and backward.

    Keys (shapes with T = batch*seq, H = hidden, F = ffn, L = seq):
      attn_x, attn_res, attn_dout [T,H], attn_bias [H]   bias+dropout+residual after attention
      ffn1_x, ffn1_dout [T,F], ffn1_bias [F]             bias+ReLU+dropout after FFN1
      ffn2_x, ffn2_res, ffn2_dout [T,H], ffn2_bias [H]   bias+dropout+residual after FFN2
      ln1_x, ln1_dy, ln2_x, ln2_dy [T,H]; ln1_gamma, ln1_beta, ln2_gamma, ln2_beta [H]
      scores, scores_dy [B, heads, L, L];  key_len [B] int32 (absent without padding)
    `which` restricts the draw to a subset of keys.
    """
    T, H, F, L, B = layer.tokens, layer.hidden, layer.ffn, layer.seq, layer.batch
    dt = layer.dtype
    spec = {
        "attn_x": ((T, H), 0.0, 1.0), "attn_res": ((T, H), 0.0, 1.0),
        "attn_dout": ((T, H), 0.0, 1.0), "attn_bias": ((H,), 0.0, 0.02),
        "ffn1_x": ((T, F), 0.0, 1.0), "ffn1_dout": ((T, F), 0.0, 1.0),
        "ffn1_bias": ((F,), 0.0, 0.02),
        "ffn2_x": ((T, H), 0.0, 1.0), "ffn2_res": ((T, H), 0.0, 1.0),
        "ffn2_dout": ((T, H), 0.0, 1.0), "ffn2_bias": ((H,), 0.0, 0.02),
        "ln1_x": ((T, H), 0.0, 1.0), "ln1_dy": ((T, H), 0.0, 1.0),
        "ln1_gamma": ((H,), 1.0, 0.1), "ln1_beta": ((H,), 0.0, 0.1),
        "ln2_x": ((T, H), 0.0, 1.0), "ln2_dy": ((T, H), 0.0, 1.0),
        "ln2_gamma": ((H,), 1.0, 0.1), "ln2_beta": ((H,), 0.0, 0.1),
        "scores": ((B, layer.heads, L, L), 0.0, 3.0),
        "scores_dy": ((B, layer.heads, L, L), 0.0, 1.0),
    }
    out = {}
    for k, (shape, mean, std) in spec.items():
        if which is None or k in which:
            out[k] = normal(seed, f"{layer.name}/{k}", shape, mean, std, dt)
    if layer.pad_lo is not None and (which is None or "key_len" in which):
        out["key_len"] = key_lengths(seed, f"{layer.name}/key_len", B, layer.pad_lo, L)
    return out


def sweep_inputs(k_len: int, seed: int = 0, elements: int = SWEEP_ELEMENTS):
    """Softmax sweep case: rows = elements / k_len rows of length k_len, laid out
    as [rows, 1, 1, k_len] (batch = rows) so each row gets its own random valid
    length U[1, k_len].  Returns (scores, scores_dy, key_len), FP16."""
    rows = elements // k_len
    shape = (rows, 1, 1, k_len)
    x = normal(seed, f"sweep{k_len}/scores", shape, 0.0, 3.0, "f16")
    dy = normal(seed, f"sweep{k_len}/scores_dy", shape, 0.0, 1.0, "f16")
    kl = key_lengths(seed, f"sweep{k_len}/key_len", rows, 1, k_len)
    return x, dy, kl


# The trainer update's workload: the parameters of a BERT-base encoder (12
# layers of H = 768, FFN = 3072, with token/position/segment embeddings, the
# embedding LayerNorm and the pooler), 109,482,240 values in one flat
# workspace.
def bert_base_param_count(layers: int = 12, hidden: int = 768, ffn: int = 3072,
                          vocab: int = 30522, positions: int = 512, segments: int = 2) -> int:
    h, f = hidden, ffn
    per_layer = 4 * h * h + 4 * h + 2 * h * f + f + h + 4 * h  # QKV+out, FFN, two LayerNorms
    embeddings = (vocab + positions + segments) * h + 2 * h
    pooler = h * h + h
    return layers * per_layer + embeddings + pooler


TRAINER_N = bert_base_param_count()


def trainer_state(n: int, seed: int = 0, dtype: str = "f16", device="cpu"):
    """Seeded trainer state of n elements, drawn with torch on `device`:
    parameters N(0, 0.02) and gradients N(0, 0.01) in the storage dtype, first
    moments N(0, 1e-3) and second moments N(0, 1e-2)^2 in FP32 (as after a few
    steps).  Returns (param, grad, exp_avg, exp_avg_sq)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(zlib.crc32(f"trainer/{seed}".encode()))
    dt = {"f16": torch.float16, "f32": torch.float32}[dtype]

    def draw(std):
        return torch.randn(n, generator=g, device=device, dtype=torch.float32) * std

    p = draw(0.02).to(dt)
    gr = draw(0.01).to(dt)
    m = draw(1e-3)
    v = draw(1e-2) ** 2
    return p, gr, m, v


# Criterion workloads: the BERT-base (30522) and GPT-2 (50257) vocabularies,
# padded to a multiple of 8 as the vectorised kernels need (30528, 50264).
CRITERION_VOCAB = {"bert-base": 30528, "gpt2-large": 50264, "transformer-base": 32000,
                   "tiny": 64}
# Embedding tables: the unpadded vocabularies (the embedding has no width
# constraint on the vocabulary).
EMBEDDING_VOCAB = {"bert-base": 30522, "gpt2-large": 50257, "transformer-base": 32000,
                   "tiny": 64}

