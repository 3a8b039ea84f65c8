"""GPU GEMM+Quantize (tcgen05 kernel) vs the CPU oracle on the same inputs.

Bars: with exactly representable products (small integers) the fp32
accumulation is exact, so the bf16 Y and every MXFP8 payload byte and E8M0
scale (compact, and packed after decoding) are bit-exact.  With N(0,1)
inputs the fp32 accumulation differs from fp64 by rounding: the bf16 Y is
within one bf16 rounding step of the oracle's Y, and an MXFP8 code or scale
may differ only where the oracle's value lies within fp32 rounding of a code
or power-of-two boundary (counted, and required to be rare and one step).
"""
import numpy as np
import pytest

import oracle
from mxfp8_block_scaled_fa_gb300 import inputs
from tests.helpers import host, to_dev, unpack_packed

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import torch
    from mxfp8_block_scaled_fa_gb300 import build, mxfa
    build.build()
    assert torch.cuda.is_available()
    return mxfa


def _operand(mx, bits, rows, K):
    """bf16 bits [rows, K] -> ROW-quantized operand with packed scales."""
    return mx.quantize(to_dev(bits.reshape(rows, K // 128, 128)), mx.ROW, mx.Seqs.dense(1, rows))


def _run(mx, a_bits, b_bits):
    import torch
    M, K = a_bits.shape
    N = b_bits.shape[0]
    a, b = _operand(mx, a_bits, M, K), _operand(mx, b_bits, N, K)
    res = mx.gemm_quant(a, b)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    return res


def _bf16(x):
    return inputs.f32_to_bf16_bits(np.asarray(x, np.float32))


def _check_packed(res, M, N, s_row, s_col):
    # the packed atoms decode (written independently in tests/helpers.py) to
    # the compact scales: ROW atoms per (128-row tile, 128-column group), COL
    # atoms likewise with 32-row blocks
    H = N // 128
    comp, pad = unpack_packed(host(res["row"].sf_packed), 0, [M], H)
    np.testing.assert_array_equal(comp, s_row)
    comp, pad = unpack_packed(host(res["col"].sf_packed), 1, [M], H)
    np.testing.assert_array_equal(comp, s_col)


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (128, 128, 128), (384, 256, 1152)])
def test_gemm_quant_exact(mx, M, N, K):
    rng = np.random.default_rng(M + N + K)
    a = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    b = rng.integers(-8, 9, size=(N, K)).astype(np.float32)
    res = _run(mx, _bf16(a), _bf16(b))
    y, (q_row, s_row), (q_col, s_col) = oracle.method_gemm_quant(a.astype(np.float64),
                                                                  b.astype(np.float64))
    np.testing.assert_array_equal(y, a.astype(np.float64) @ b.astype(np.float64).T)
    np.testing.assert_array_equal(host(res["bf16"].view(__import__("torch").int16)).view(np.uint16),
                                  _bf16(y))
    np.testing.assert_array_equal(host(res["row"].data), q_row)
    np.testing.assert_array_equal(host(res["row"].sf_compact), s_row)
    np.testing.assert_array_equal(host(res["col"].data), q_col)
    np.testing.assert_array_equal(host(res["col"].sf_compact), s_col)
    _check_packed(res, M, N, s_row, s_col)


def test_gemm_quant_normal_inputs(mx):
    import torch
    M, N, K = 512, 256, 1024
    a_bits = inputs.normal_bf16((M, K), 11)
    b_bits = inputs.normal_bf16((N, K), 12)
    res = _run(mx, a_bits, b_bits)
    f = lambda x: inputs.bf16_bits_to_f32(x).astype(np.float64)
    y, (q_row, s_row), (q_col, s_col) = oracle.method_gemm_quant(f(a_bits), f(b_bits))
    yb = f(host(res["bf16"].view(torch.int16)).view(np.uint16))
    # one bf16 rounding step of the oracle's value, plus the fp32 sum's error
    e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -126)))
    assert np.all(np.abs(yb - y) <= 2.0 ** (e - 8) + 1e-5 * np.abs(y) + 1e-6)
    for name, q, s in (("row", q_row, s_row), ("col", q_col, s_col)):
        gq, gs = host(res[name].data), host(res[name].sf_compact)
        # scales: only a block maximum within fp32 rounding of a power of two may differ
        assert np.mean(gs != s) <= 1e-3, (name, np.mean(gs != s))
        same = (np.repeat(gs, 32, axis=1) == np.repeat(s, 32, axis=1)) if name == "row" else \
            (np.repeat(gs, 32, axis=0) == np.repeat(s, 32, axis=0))
        diff = (gq != q) & same
        assert np.mean(diff) <= 1e-3, (name, np.mean(diff))
        # differing codes are neighbours (one step of the E4M3 grid)
        gv, ov = oracle.e4m3_decode(gq[diff][:200]), oracle.e4m3_decode(q[diff][:200])
        assert np.all(np.abs(gv - ov) <= np.abs(ov) / 8 + 2.0 ** -9), name
    _check_packed(res, M, N, host(res["row"].sf_compact), host(res["col"].sf_compact))


def test_tensor_peak_probe(mx):
    # the calibration kernel behind the benchmark's roofline peak: every CTA
    # reports its cycles, and the rate per SM stays at or below the dense
    # MXFP8 MMA rate (8192 E4M3 MACs per clock per SM on this GPU)
    import torch
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    cyc = torch.zeros(nsm, dtype=torch.int64, device="cuda")
    mx.mxfa_tensor_peak_probe(256, nsm, cyc)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    c = host(cyc).astype(np.float64)
    assert np.all(c > 0)
    rate = 256 * 4 * 128 * 256 * 32 / c
    assert np.all(rate <= 8192 * 1.01) and np.all(rate >= 2048), rate.min()


def test_gemm_quant_nan_rows(mx):
    # a NaN in one element of A makes its quantized block NaN (scale 0xFF), so
    # that row of Y is NaN: its ROW blocks and the COL blocks holding it carry
    # scale 0xFF and 0x7F payloads; every other row is exact
    M, N, K = 256, 256, 256
    rng = np.random.default_rng(77)
    a = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    b = rng.integers(-8, 9, size=(N, K)).astype(np.float32)
    a[37, 5] = np.nan
    res = _run(mx, _bf16(a), _bf16(b))
    ad = a.astype(np.float64)
    ad[37, :32] = np.nan  # the whole quantized block of A reads as NaN
    y, (q_row, s_row), (q_col, s_col) = oracle.method_gemm_quant(ad, b.astype(np.float64))
    assert np.isnan(y[37]).all() and not np.isnan(np.delete(y, 37, axis=0)).any()
    np.testing.assert_array_equal(host(res["row"].sf_compact), s_row)
    np.testing.assert_array_equal(host(res["row"].data), q_row)
    np.testing.assert_array_equal(host(res["col"].sf_compact), s_col)
    np.testing.assert_array_equal(host(res["col"].data), q_col)
    assert np.all(host(res["row"].sf_compact)[37] == 0xFF) and np.all(host(res["col"].sf_compact)[1] == 0xFF)
    _check_packed(res, M, N, s_row, s_col)
