"""The oracle's projection GEMM (fp64 y = a b^T), pinned by a hand-worked case
and by numpy's matmul, and its GEMM+Quantize step by the quantizer's own pins
applied to a product whose value is known exactly (CPU only)."""
import numpy as np

import oracle


def test_gemm_hand_worked():
    # a = [[1, 2], [3, 4]], b = [[5, 6], [7, 8]] (rows = output features):
    # y = a b^T = [[1*5 + 2*6, 1*7 + 2*8], [3*5 + 4*6, 3*7 + 4*8]] = [[17, 23], [39, 53]]
    a = np.array([[1.0, 2.0], [3.0, 4.0]])
    b = np.array([[5.0, 6.0], [7.0, 8.0]])
    np.testing.assert_array_equal(oracle.gemm_nt(a, b), [[17.0, 23.0], [39.0, 53.0]])


def test_gemm_equals_library_matmul():
    rng = np.random.default_rng(0)
    a = rng.standard_normal((37, 96))
    b = rng.standard_normal((21, 96))
    np.testing.assert_allclose(oracle.gemm_nt(a, b), a @ b.T, rtol=1e-12, atol=1e-12)


def test_gemm_quant_exact_products():
    # integer inputs up to 8 are exact in E4M3 under any block scale the rule
    # picks, so the quantized GEMM's Y is the exact integer product, and its
    # ROW / COL outputs are the quantizer applied to that exact Y
    rng = np.random.default_rng(1)
    a = rng.integers(-8, 9, size=(64, 128)).astype(np.float64)
    b = rng.integers(-8, 9, size=(32, 128)).astype(np.float64)
    y, row, col = oracle.method_gemm_quant(a, b)
    np.testing.assert_array_equal(y, a @ b.T)
    for got, mode in ((row, oracle.ROW), (col, oracle.COL)):
        q, s = oracle.quantize(a @ b.T, mode)
        np.testing.assert_array_equal(got[0], q)
        np.testing.assert_array_equal(got[1], s)
    # a block whose maximum is 448: scale 2^(8 - 8) and payload 448 -> 0x7E
    yq, sq = oracle.quantize(np.full((1, 32), 448.0), oracle.ROW)
    assert sq[0, 0] == 127 and np.all(yq == 0x7E)
