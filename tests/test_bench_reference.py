"""The benchmark's SQNR reference (fp64 attention without quantization on the
host, chunked over query rows) agrees with the oracle's unquantized attention
and gradients, causal and not, across chunk boundaries (CPU only)."""
import importlib.util
import math
import os
import sys

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


@pytest.mark.parametrize("causal,lq,lk", [(False, 300, 200), (True, 300, 300)])
def test_exact_attention_matches_oracle(bench, causal, lq, lk):
    import torch
    rng = np.random.default_rng(7)
    q, do = rng.standard_normal((lq, 128)), rng.standard_normal((lq, 128))
    k, v = rng.standard_normal((lk, 128)), rng.standard_normal((lk, 128))
    scale = 1 / math.sqrt(128)
    got = bench.exact_attention(torch, q, k, v, do, scale, causal, chunk=128)
    o, lse = oracle.method_fwd(q[:, None], k[:, None], v[:, None], None, None, scale, causal, False)
    g = oracle.method_bwd(q[:, None], k[:, None], v[:, None], do[:, None], o, lse, None, None, scale,
                          causal, False)
    for a, b in zip([o] + list(g), got):
        np.testing.assert_allclose(b, a.reshape(b.shape), rtol=0, atol=1e-12)


def test_sqnr_db(bench):
    r = np.ones((4, 4))
    # noise power 1/100 of the signal -> 20 dB; a missing output is skipped
    out = bench.sqnr_db([r * 1.1, None], [r, r])
    assert out == {"O": pytest.approx(20.0)}
