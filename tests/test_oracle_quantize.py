"""Pins for the oracle's block orientations and segment anchoring (CPU only)."""
import numpy as np

import oracle
from mxfp8_block_scaled_fa_gb300 import inputs


def _x(rows, cols, seed):
    b = inputs.normal_bf16((rows, cols), seed)
    return inputs.bf16_bits_to_f32(b).astype(np.float64)


def test_col_is_row_of_transpose():
    # 32x1 blocks along rows are 1x32 blocks of the transposed matrix
    x = _x(96, 64, 1)
    qc, sc = oracle.quantize(x, oracle.COL)
    qr, sr = oracle.quantize(x.T.copy(), oracle.ROW)
    np.testing.assert_array_equal(qc, qr.T)
    np.testing.assert_array_equal(sc, sr.T)


def test_square_is_transpose_invariant():
    # the same payload serves both orientations (one scale per 32x32 block)
    x = _x(128, 96, 2)
    q, s = oracle.quantize(x, oracle.SQ)
    qt, st = oracle.quantize(x.T.copy(), oracle.SQ)
    np.testing.assert_array_equal(q, qt.T)
    np.testing.assert_array_equal(s, st.T)


def test_square_scale_is_max_of_row_scales():
    # the square block's amax is the max of its 32 row-block amaxes, and the
    # E8M0 byte is monotone in amax
    x = _x(64, 64, 3)
    _, ssq = oracle.quantize(x, oracle.SQ)
    _, srow = oracle.quantize(x, oracle.ROW)
    for rb in range(2):
        for cb in range(2):
            assert ssq[rb, cb] == srow[rb * 32:(rb + 1) * 32, cb].max()


def test_segments_anchor_blocks():
    # ragged segments quantize exactly as if each were quantized alone
    lens = [45, 32, 7, 70]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = _x(int(cu[-1]), 64, 4)
    for mode in (oracle.COL, oracle.SQ):
        q, s = oracle.quantize(x, mode, cu)
        srow = 0
        for g, n in enumerate(lens):
            qg, sg = oracle.quantize(x[cu[g]:cu[g + 1]], mode)
            np.testing.assert_array_equal(q[cu[g]:cu[g + 1]], qg)
            nb = (n + 31) // 32
            np.testing.assert_array_equal(s[srow:srow + nb], sg)
            srow += nb
        assert srow == s.shape[0] == oracle.sf_rows(cu, int(cu[-1]))


def test_partial_block_uses_only_its_rows():
    # a trailing 7-row column block: scale from those 7 rows only
    x = np.zeros((7, 32))
    x[:, 0] = 1.0
    x[3, 0] = 5.0  # floor(log2 5) = 2 -> byte 121
    q, s = oracle.quantize(x, oracle.COL)
    assert s.shape == (1, 32)
    assert s[0, 0] == 121 and s[0, 1] == 0
