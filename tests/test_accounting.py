"""Pins the byte and roofline arithmetic that bench.py reports against the
worked examples the pages print (tests/golden/pages_worked_examples.json),
and checks the per-operator byte counts against hand counts."""
import json
import os

import numpy as np
import pytest

from transformer_layer_non_gb300 import accounting as acc

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "pages_worked_examples.json")))


def test_three_matrix_add_traffic():
    g = GOLDEN["three_matrix_add"]
    size = 1000.0
    unfused = acc.unfused_chain_traffic(3, size)
    fused = acc.traffic([size] * 3, [size])
    assert unfused == (g["unfused"]["reads"] + g["unfused"]["writes"]) * size
    assert fused == (g["fused"]["reads"] + g["fused"]["writes"]) * size


def test_fused_ln_gelu_dropout_traffic():
    g = GOLDEN["ln_gelu_dropout_fusion"]
    s = 4096.0
    three_kernels = sum(acc.traffic([s], [s]) for _ in range(3))
    one_kernel = acc.traffic([s], [s])
    assert three_kernels / s == g["unfused_traffic_in_units_of_size_x"]
    assert one_kernel / s == g["fused_traffic_in_units_of_size_x"]


def test_arithmetic_intensity_examples():
    g = GOLDEN["gemm_8192_bf16"]
    n, b = g["N"], g["bytes_per_element"]
    nbytes = acc.traffic([n * n * b, n * n * b], [n * n * b])
    flops = 2.0 * n**3
    assert nbytes == pytest.approx(g["bytes_approx"], rel=0.01)
    assert flops == pytest.approx(g["flops_approx"], rel=0.01)
    assert acc.arithmetic_intensity(flops, nbytes) == pytest.approx(g["ai_approx"], rel=0.02)
    g2 = GOLDEN["elementwise_add_8192_bf16"]
    ai = acc.arithmetic_intensity(float(n * n), nbytes)
    assert n * n == pytest.approx(g2["flops_approx"], rel=0.01)
    assert ai == pytest.approx(g2["ai_approx"], rel=0.02)


def test_ridge_point_and_attainable():
    g = GOLDEN["h100_ridge_point"]
    r = acc.ridge_point(g["peak_flops"], g["bandwidth_bytes_per_s"])
    assert r == pytest.approx(g["ridge_approx"], rel=0.01)
    assert acc.attainable(g["peak_flops"], g["bandwidth_bytes_per_s"], 0.17) == pytest.approx(
        0.17 * g["bandwidth_bytes_per_s"])
    assert acc.attainable(g["peak_flops"], g["bandwidth_bytes_per_s"], 2700) == g["peak_flops"]


def test_operator_bytes_by_hand():
    # BERT-base bias+dropout+residual forward: 4096 x 768 FP16; reads x and
    # residual (2 B each), writes out (2 B) and one mask bit per element.
    n = 4096 * 768
    assert acc.bdr_fwd_bytes(4096, 768, 2) == n * 6.125 + 768 * 2
    assert acc.dropout_bwd_bytes(4096, 768, 2) == n * 4.125 + 768 * 2
    assert acc.brd_fwd_bytes(4096, 3072, 2) == 4096 * 3072 * 4.125 + 3072 * 2
    assert acc.ln_fwd_bytes(4096, 768, 2) == n * 4 + 2 * 768 * 2 + 8 * 4096
    assert acc.ln_bwd_bytes(4096, 768, 2) == n * 6 + 3 * 768 * 2 + 8 * 4096


def test_softmax_valid_counts():
    # causal square: q sees q+1 keys -> L(L+1)/2 per head
    assert acc.softmax_valid_count(1, 1, 4, 4, None, True) == 10
    # padding: min(key_len, k_len) per query
    assert acc.softmax_valid_count(2, 3, 5, 8, np.array([3, 20]), False) == 3 * 5 * (3 + 8)
    # causal and padding together, q_len < k_len (bottom-right diagonal)
    kl = np.array([2])
    # q=0 sees j<=2 -> 3 keys, capped at 2; q=1 -> 4 keys capped at 2
    assert acc.softmax_valid_count(1, 1, 2, 4, kl, True) == 4
    # negative key lengths count as zero valid keys
    assert acc.softmax_valid_count(1, 1, 2, 8, np.array([-1]), False) == 0
    v = acc.softmax_valid_count(1, 1, 1, 16, np.array([7]), False)
    assert acc.softmax_fwd_bytes(1, 1, 1, 16, 2, np.array([7])) == v * 2 + 4 + 16 * 2
    assert acc.softmax_bwd_bytes(1, 1, 1, 16, 2, np.array([7])) == v * 4 + 4 + 16 * 2


def test_next_operator_bytes_by_hand():
    # [4, 96] QKV rows: 384 values in and out, plus the 96-value bias.
    assert acc.qkv_fwd_bytes(4, 96, 2) == 384 * 2 * 2 + 96 * 2
    assert acc.qkv_bwd_bytes(4, 96, 2) == 384 * 2 * 2 + 96 * 2
    # Trainer: 22 bytes per FP16 element (2+2+4+4 in, 2+4+4 out).
    assert acc.adam_bytes(1000, 2) == 22000
    # Softmax+dropout over [1, 1, 2, 16] with 8 valid keys per row: 16 valid
    # values in; 2 x 32 values and 32 mask bits out.
    kl = np.array([8], dtype=np.int32)
    assert acc.softmax_dropout_fwd_bytes(1, 1, 2, 16, 2, kl) == 16 * 2 + 4 + 2 * 32 * 2 + 4
    assert acc.softmax_dropout_bwd_bytes(1, 1, 2, 16, 2, kl) == 2 * 16 * 2 + 2 + 4 + 32 * 2
    # Cross entropy over [3, 64]: the logits once (+ per-row FP32/int32 values).
    assert acc.cross_entropy_fwd_bytes(3, 64, 2) == 3 * 64 * 2 + 12 + 24
    assert acc.cross_entropy_bwd_bytes(3, 64, 2) == 2 * 3 * 64 * 2 + 36
    # Embedding: 10 tokens of width 16 at seq 5, 4 distinct ids.
    assert acc.embedding_fwd_bytes(10, 5, 16, 2) == 40 + 320 + 160 + 320 + 20
    assert acc.embedding_bwd_bytes(10, 4, 16, 2) == 40 + 320 + 20 + 2 * 256



def test_read_write_split_adds_up_to_the_step_bytes():
    from transformer_layer_non_gb300 import synth

    for L in synth.LAYERS.values():
        es = 2 if L.dtype == "f16" else 4
        kl = synth.layer_inputs(L, 0, which={"key_len"}).get("key_len")
        tot = acc.layer_step_bytes(L.tokens, L.hidden, L.ffn, L.batch, L.heads, L.seq, es,
                                          kl, L.causal)
        rw = acc.layer_step_read_write(L.tokens, L.hidden, L.ffn, L.batch, L.heads, L.seq,
                                              es, kl, L.causal)
        assert set(rw) == set(tot)
        for k in tot:
            assert abs(sum(rw[k]) - tot[k]) <= 1e-6 * tot[k], (L.name, k)
