"""Pins for the oracle's dropout generator (Philox-4x32-10) and keep rule.

The pages name no generator; the kernels and the oracle each implement
Philox-4x32-10 from Salmon et al., "Parallel Random Numbers: As Easy as 1, 2,
3" (SC'11).  The oracle's copy is pinned here against an implementation that
is not ours: libtorch's header-only ``at::philox_engine`` (compiled from the
installed headers into a tiny probe), and by the statistics of the keep rule.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle


def _torch_include():
    try:
        import torch.utils.cpp_extension as ce
    except Exception:  # pragma: no cover
        return None
    for p in ce.include_paths():
        if os.path.exists(os.path.join(p, "ATen", "core", "PhiloxRNGEngine.h")):
            return p
    return None


_PROBE = r"""
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdio>
int main() {
  unsigned long long seed, subseq, off;
  while (std::scanf("%llu %llu %llu", &seed, &subseq, &off) == 3) {
    at::philox_engine e(seed, subseq, off);
    for (int k = 0; k < 4; ++k) std::printf("%u ", e());
    std::printf("\n");
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def torch_philox(tmp_path_factory):
    inc = _torch_include()
    if inc is None or shutil.which("g++") is None:
        pytest.skip("libtorch headers or g++ not available")
    d = tmp_path_factory.mktemp("philox_probe")
    src = d / "probe.cpp"
    src.write_text(_PROBE)
    exe = d / "probe"
    subprocess.run(["g++", "-std=c++17", "-O1", f"-I{inc}", str(src), "-o", str(exe)], check=True)

    def run(triples):
        inp = "".join(f"{s} {u} {o}\n" for s, u, o in triples)
        out = subprocess.run([str(exe)], input=inp, capture_output=True, text=True, check=True)
        return [[int(v) for v in line.split()] for line in out.stdout.strip().splitlines()]

    return run


def test_philox_matches_libtorch_engine(torch_philox):
    # libtorch's engine(seed, subsequence, offset) yields the four words of
    # counter block `offset` in stream `subsequence`; in our convention the
    # stream is the call's dropout offset and the block is element index >> 2.
    rng = np.random.default_rng(1234)
    triples = [(0, 0, 0), (1, 0, 0), (0, 1, 0), (0, 0, 1),
               (2**64 - 1, 2**64 - 1, 2**62 - 1),   # every key/stream bit; largest block of a 64-bit index
               (0xDEADBEEF, 2**32, 2**32 + 5),          # high counter words in use
               (2**63 + 17, 3, 2**40 + 1)]
    for _ in range(200):
        triples.append((int(rng.integers(0, 2**63)), int(rng.integers(0, 2**40)),
                        int(rng.integers(0, 2**40))))
    ref = torch_philox(triples)
    for (seed, stream, block), words in zip(triples, ref):
        ours = [oracle.dropout_word(seed, stream, 4 * block + k) for k in range(4)]
        assert ours == words, (seed, stream, block)


def test_philox_block_function_is_the_word_source():
    # dropout_word(seed, offset, i) is word i&3 of Philox(ctr=(i>>2, offset), key=seed).
    seed, off = 0x0123456789ABCDEF, 0xFEDCBA9876543210
    for i in [0, 1, 2, 3, 4, 5, 2**32 * 4 + 2, 2**40 + 7]:
        blk = i >> 2
        out = oracle.philox4x32_10([blk & 0xFFFFFFFF, blk >> 32, off & 0xFFFFFFFF, off >> 32],
                                   [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.dropout_word(seed, off, i) == int(out[i & 3])


def test_threshold_rule():
    assert oracle.dropout_threshold(0.0) == 0
    assert oracle.dropout_threshold(1e-12) == 0          # below one part in 2^32
    assert oracle.dropout_threshold(0.5) == 2**31
    assert oracle.dropout_threshold(0.25) == 2**30
    p = np.float32(0.1)
    assert oracle.dropout_threshold(float(p)) == int(np.floor(float(p) * 2.0**32))
    assert oracle.dropout_threshold(float(np.nextafter(np.float32(1), np.float32(0)))) < 2**32


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_keep_fraction_within_3_sigma(p):
    n = 1 << 20
    words = oracle.dropout_keep_bits(n, p, seed=0, offset=11)
    kept = int(np.unpackbits(words.view(np.uint8)).sum())
    sigma = np.sqrt(p * (1 - p) / n)
    assert abs(kept / n - (1 - p)) <= 3 * sigma


def test_p_zero_keeps_all_and_tail_bits_are_zero():
    n = 70  # 2 full words and 6 bits of a third
    w = oracle.dropout_keep_bits(n, 0.0, seed=3, offset=4)
    assert w.shape == (3,)
    assert w[0] == 0xFFFFFFFF and w[1] == 0xFFFFFFFF and w[2] == (1 << 6) - 1


def test_streams_are_distinct():
    # Different offsets (call sites) and seeds must give different masks.
    a = oracle.dropout_keep_bits(4096, 0.5, seed=0, offset=0)
    b = oracle.dropout_keep_bits(4096, 0.5, seed=0, offset=1)
    c = oracle.dropout_keep_bits(4096, 0.5, seed=1, offset=0)
    agree_ab = np.unpackbits((~(a ^ b)).view(np.uint8)).mean()
    agree_ac = np.unpackbits((~(a ^ c)).view(np.uint8)).mean()
    assert 0.45 < agree_ab < 0.55 and 0.45 < agree_ac < 0.55
