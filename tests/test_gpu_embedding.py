"""GPU parity: the embedding layer against the FP64 oracle through the C ABI.
Forward: keep bits bit-exact, values within |err| <= 2e-3 + 2e-3*|ref|.
Backward (a deterministic scatter-add into an FP32 table gradient): within
the same bound and within the FP32 summation error bound of each row's terms,
bit-identical from run to run, and accumulated into what the table gradient
held.  Cases: the layer shapes with
BERT/GPT-2 vocabularies, uniform and word-frequency-like (Zipf) ids, a tiny
vocabulary (long runs of repeated ids), one id on 30% of the tokens, ids past
16 bits (FP16 and FP32 rows), the largest token count per call (ids spread,
and all on one id), a single token, no id in the table, rows wider than one
pass of column vectors, ragged token counts and ids outside the table."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import Guarded, assert_close, dev, f64, require_gpu, tdtype
from transformer_layer_non_gb300 import ls_ops, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

P_DROP, SEED, OFF = 0.1, 99, 4


def _case(B, L, H, V, dtype, seed=0, bad_ids=False, skew=False):
    rng = np.random.default_rng(seed)
    tok = rng.integers(0, V, B * L).astype(np.int32)
    if skew == "zipf":  # word-frequency-like ids: a few hundred repeats of the commonest
        tok = ((rng.zipf(1.1, B * L) - 1) % V).astype(np.int32)
    elif skew == "one":  # every token on one id
        tok[:] = V - 1
    elif skew == "none":  # every id outside the table
        tok[:] = np.where(rng.random(B * L) < 0.5, -1 - tok, V + tok)
    elif skew:  # a padding-like id on 30% of the tokens: one run of ~0.3*B*L rows
        tok[rng.random(B * L) < 0.3] = 0
    if bad_ids:
        tok[::13] = -1
        tok[5::17] = V + 3
    E = synth.normal(seed, f"emb{V}x{H}/E", (V, H), 0.0, 1.0, dtype)
    P = synth.normal(seed, f"emb{L}x{H}/P", (L + 2, H), 0.0, 1.0, dtype)
    dy = synth.normal(seed, f"emb{B}x{L}x{H}/dy", (B * L, H), 0.0, 1.0, dtype)
    return tok, E, P, dy


@pytest.mark.parametrize("B,L,H,V,dtype,bad,skew", [
    (2, 16, 64, 50, "f32", False, False),
    (3, 37, 24, 5, "f16", True, False),        # 111 tokens, 5 ids: long runs
    (8, 512, 768, 30522, "f16", False, False),  # BERT-base
    (8, 512, 768, 30522, "f16", False, True),   # BERT-base, one id on 30% of the tokens
    (4, 1024, 1280, 50257, "f16", True, False),  # GPT-2-large, some ids outside the table
    (2, 100, 4104, 300, "f32", False, True),    # H past one pass of column vectors per lane
    (8, 512, 768, 30522, "f16", False, "zipf"),  # BERT-base, word-frequency-like ids
    (4, 1024, 1280, 50257, "f16", False, "zipf"),  # GPT-2-large, word-frequency-like ids
    (3, 250, 136, 70000, "f16", True, "zipf"),  # ids past 16 bits
    (16, 1024, 64, 1000, "f16", False, False),  # the most tokens one call takes, ~16 per id
    (1, 16384, 16, 3, "f16", False, "one"),     # the most tokens, all on one id
    (1, 1, 8, 3, "f16", False, False),          # one token, one column vector
    (3, 5, 40, 20, "f16", False, "none"),       # no id in the table: no gradient
    (2, 300, 72, 90000, "f32", True, "zipf"),   # FP32 rows, ids past 16 bits
])
def test_forward_and_backward(B, L, H, V, dtype, bad, skew):
    require_gpu()
    tok, E, P, dy = _case(B, L, H, V, dtype, seed=H, bad_ids=bad, skew=skew)
    s = float(np.sqrt(H))
    T = B * L
    y = Guarded((T, H), tdtype(E.dtype))
    m = Guarded(((T * H + 31) // 32,), torch.int32)
    ls_ops.ls_embedding_fwd(y.t, m.t, dev(tok), dev(E), dev(P), B, L, s, P_DROP, SEED, OFF)
    torch.cuda.synchronize()
    y.check()
    m.check()
    ry, rw = oracle.embedding_fwd(tok, E, P, B, L, float(np.float32(s)), P_DROP, SEED, OFF)
    np.testing.assert_array_equal(m.t.cpu().numpy().view(np.uint32), rw, "keep bits")
    assert_close(f64(y.t), ry, "y")

    base = synth.normal(1, f"emb{V}x{H}/dE0", (V, H), 0.0, 0.01, "f32")
    ws = torch.empty(ls_ops.embedding_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        dE = dev(base)
        ls_ops.ls_embedding_bwd(dE, dev(dy), m.t, dev(tok), B, L, s, P_DROP, workspace=ws)
        torch.cuda.synchronize()
        outs.append(dE.cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])  # deterministic
    ref = oracle.embedding_bwd(tok, dy, rw, V, float(np.float32(s)), P_DROP, dE=base)
    assert_close(outs[0].astype(np.float64), ref, "dE")
    bound = _sum_bound(tok, dy, rw, V, s, base)
    _within(outs[0], ref, bound, "dE")
    # The pages' atomic mode: the same sums up to the order of the additions.
    dE = dev(base)
    ls_ops.ls_embedding_bwd(dE, dev(dy), m.t, dev(tok), B, L, s, P_DROP, deterministic=False)
    torch.cuda.synchronize()
    got = dE.cpu().numpy()
    assert_close(got.astype(np.float64), ref, "dE (atomic)")
    _within(got, ref, bound, "dE (atomic)")


def _sum_bound(tok, dy, rw, V, s, base):
    """Error bound of an FP32 sum of a row's n terms into base, in any order:
    |computed - exact| <= (n + 2) u (sum of |terms| + |base|), u = 2^-24 (the
    recursive-summation bound, one more rounding for each scaled term and one
    for the final add), doubled as margin."""
    absum = oracle.embedding_bwd(tok, np.abs(dy), rw, V, float(np.float32(s)), P_DROP,
                                 dE=np.zeros_like(base))
    ok = (tok >= 0) & (tok < V)
    n = np.bincount(tok[ok], minlength=V)[:V].astype(np.float64)[:, None]
    return 2.0 * (n + 2.0) * 2.0 ** -24 * (absum + np.abs(base.astype(np.float64)))


def _within(got, ref, bound, what):
    err = np.abs(got.astype(np.float64) - ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements past the summation bound, "
                           f"worst err {err[bad].max():.3g} vs bound {bound[bad].min():.3g}")
