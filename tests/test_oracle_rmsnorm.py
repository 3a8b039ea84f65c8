"""Pins for the oracle's fused RMSNorm + Quantize (CPU only).

y = (x * r) * gamma with r = 1/sqrt(mean(x^2) + eps), computed in the fused
kernel's fp32 order; the quantized codes then follow the pinned MX quantizer.
"""
import numpy as np

import oracle
from mxfp8_block_scaled_fa_gb300 import inputs


def test_close_to_fp64_definition():
    x = inputs.bf16_bits_to_f32(inputs.normal_bf16((64, 2048), 1))
    g = np.random.default_rng(2).uniform(0.5, 1.5, 2048).astype(np.float32)
    out = oracle.rmsnorm_quant(x, g, 1e-6, 7, 8192, want_y=True)
    x64 = x.astype(np.float64)
    r = 1.0 / np.sqrt(np.mean(x64 * x64, axis=1, keepdims=True) + 1e-6)
    y64 = x64 * r * g.astype(np.float64)
    rel = np.abs(out["y"] - y64) / np.maximum(np.abs(y64), 1e-30)
    assert rel.max() < 4e-7  # a few fp32 roundings


def test_summation_order_is_the_documented_one():
    # C = 256: lane 0 owns columns 0..7.  Adding 2^24 (x = 2^12) first and
    # then seven 1.0 squares loses every 1 (2^24 + 1 rounds back to 2^24), so
    # sumsq = 2^24 exactly, mean = 2^16, mean + 1e-6 rounds to 2^16, r = 2^-8:
    # y0 = 2^12 * 2^-8 = 16 and y1..7 = 2^-8 exactly (gamma = 1).  The exact
    # sum (2^24 + 7) would give y0 = 15.99999666...
    x = np.zeros((1, 256), np.float32)
    x[0, 0] = 4096.0
    x[0, 1:8] = 1.0
    g = np.ones(256, np.float32)
    y = oracle.rmsnorm_quant(x, g, 1e-6, 1, 8192, want_y=True)["y"]
    assert y[0, 0] == 16.0
    assert np.all(y[0, 1:8] == 2.0 ** -8)
    assert np.all(y[0, 8:] == 0.0)


def test_constant_rows_closed_form():
    # rows of +-1: sumsq = C exactly, mean = 1, r = fl(1 / fl(sqrt(fl(1 + eps))))
    x = np.where(np.arange(2048) % 3 == 0, -1.0, 1.0).astype(np.float32)[None, :]
    x = np.repeat(x, 32, axis=0)
    g = np.full(2048, 0.75, np.float32)
    y = oracle.rmsnorm_quant(x, g, 1e-6, 1, 8192, want_y=True)["y"]
    one = np.float32(1.0)
    r = one / np.sqrt(one + np.float32(1e-6))
    expect = (x * r) * g
    np.testing.assert_array_equal(y, expect)


def test_outputs_are_the_quantized_y():
    x = inputs.bf16_bits_to_f32(inputs.normal_bf16((96, 512), 3))
    g = np.random.default_rng(4).uniform(0.5, 1.5, 512).astype(np.float32)
    out = oracle.rmsnorm_quant(x, g, 1e-6, 7, 64, want_y=True)
    y = out["y"].astype(np.float64)
    cu = np.array([0, 64, 96], np.int32)
    for key, mode in (("row", oracle.ROW), ("col", oracle.COL), ("sq", oracle.SQ)):
        q, s = oracle.quantize(y, mode, cu)
        np.testing.assert_array_equal(out[key][0], q)
        np.testing.assert_array_equal(out[key][1], s)
