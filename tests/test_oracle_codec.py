"""Pins for the oracle's E4M3 / E8M0 codecs and block quantizer (CPU only).

Each check is tied to something other than the oracle itself: the OCP E4M3
format facts (bias 7, largest finite 448, smallest subnormal 2^-9, NaN at
0x7F/0xFF, no infinity), hand-worked examples in tests/golden/, and algebraic
properties of a power-of-two block scale.
"""
import math
import os
import re

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_quant_blocks.txt")

_NUM = re.compile(r"^-?\d+(\.\d+)?(\*2\*\*-?\d+)?$|^-?2\*\*-?\d+$|^-0\.0$")


def _val(s: str) -> float:
    s = s.strip()
    assert _NUM.match(s), f"unexpected literal {s!r}"
    neg = s.startswith("-")
    body = s[1:] if neg else s
    if body.startswith("2**"):
        v = 2.0 ** int(body[3:])
    elif "*2**" in body:
        a, b = body.split("*2**")
        v = float(a) * 2.0 ** int(b)
    else:
        v = float(body)
    return -v if neg else v


def _golden_cases():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = [p.strip() for p in line.split(";")]
        name = f[0]
        kv = dict(p.split("=", 1) for p in f[1:])
        x = np.full(32, _val(kv["rest"]))
        for item in filter(None, kv["values"].split(",")):
            i, v = item.split(":")
            x[int(i)] = _val(v)
        codes = np.full(32, int(kv["rest_code"], 16), np.uint8)
        for item in filter(None, kv["codes"].split(",")):
            i, c = item.split(":")
            codes[int(i)] = int(c, 16)
        cases.append((name, x, int(kv["sf"], 16), codes))
    assert len(cases) >= 10
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_golden_blocks(case):
    name, x, sf, codes = case
    q, s = oracle.quantize(x.reshape(1, 32), oracle.ROW)
    assert s[0, 0] == sf, name
    np.testing.assert_array_equal(q[0], codes, err_msg=name)


def test_e4m3_format_facts():
    # OCP E4M3: bias 7, 3 mantissa bits, largest finite 448 (0x7E), smallest
    # subnormal 2^-9 (0x01), smallest normal 2^-6 (0x08), 1.0 = 0x38, NaN 0x7F.
    assert oracle.e4m3_decode([0x7E])[0] == 448.0
    assert oracle.e4m3_decode([0x01])[0] == 2.0 ** -9
    assert oracle.e4m3_decode([0x08])[0] == 2.0 ** -6
    assert oracle.e4m3_decode([0x07])[0] == 7 * 2.0 ** -9
    assert oracle.e4m3_decode([0x38])[0] == 1.0
    assert oracle.e4m3_decode([0xB8])[0] == -1.0
    assert math.isnan(oracle.e4m3_decode([0x7F])[0])
    assert math.isnan(oracle.e4m3_decode([0xFF])[0])
    pos = oracle.e4m3_decode(np.arange(0x00, 0x7F))
    assert np.all(np.diff(pos) > 0)  # codes 0x00..0x7E strictly increasing
    # each normal binade [2^e, 2^(e+1)) holds exactly 8 codes
    for e in range(-6, 9):
        n = np.sum((pos >= 2.0 ** e) & (pos < 2.0 ** (e + 1)))
        assert n == (7 if e == 8 else 8), e  # 0x7F (would be 480) is NaN


def test_e4m3_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes)
    back = oracle.e4m3_encode(vals)
    np.testing.assert_array_equal(back, codes)


def test_e4m3_rounding_midpoints_and_saturation():
    pos = oracle.e4m3_decode(np.arange(0x00, 0x7F))
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2
    enc = oracle.e4m3_encode(mid)
    codes_lo = np.arange(0x00, 0x7E)
    # ties go to the even code (mantissa LSB 0)
    expect = np.where(codes_lo % 2 == 0, codes_lo, codes_lo + 1)
    np.testing.assert_array_equal(enc, expect.astype(np.uint8))
    eps = 1e-9
    np.testing.assert_array_equal(oracle.e4m3_encode(mid * (1 - eps)), codes_lo)
    np.testing.assert_array_equal(oracle.e4m3_encode(mid * (1 + eps)), codes_lo + 1)
    for big in (448.0, 463.9, 464.0, 1e6, float("inf")):
        assert oracle.e4m3_encode([big])[0] == 0x7E
        assert oracle.e4m3_encode([-big])[0] == 0xFE
    assert oracle.e4m3_encode([float("nan")])[0] == 0x7F


def test_e8m0_bit_extraction():
    # E8M0 byte = exponent of amax - 8 + 127, clamped to [0, 254]
    assert oracle.e8m0_from_amax(1.0) == 119
    assert oracle.e8m0_from_amax(1.9999) == 119
    assert oracle.e8m0_from_amax(2.0) == 120
    assert oracle.e8m0_from_amax(448.0) == 127  # floor(log2 448) = 8
    assert oracle.e8m0_from_amax(0.0) == 0
    assert oracle.e8m0_from_amax(2.0 ** -119) == 0
    assert oracle.e8m0_from_amax(2.0 ** -118) == 1
    assert oracle.e8m0_from_amax(float("nan")) == 0xFF
    assert oracle.e8m0_from_amax(float("inf")) == 0xFF
    assert oracle.e8m0_decode(127) == 1.0
    assert oracle.e8m0_decode(0) == 2.0 ** -127
    assert math.isnan(oracle.e8m0_decode(0xFF))


def test_nonfinite_block():
    x = np.ones((1, 32))
    x[0, 5] = np.nan
    q, s = oracle.quantize(x, oracle.ROW)
    assert s[0, 0] == 0xFF and np.all(q == 0x7F)
    x[0, 5] = np.inf
    q, s = oracle.quantize(x, oracle.ROW)
    assert s[0, 0] == 0xFF and np.all(q == 0x7F)


def _bf16_exact(rng, n, scale=1.0):
    from mxfp8_block_scaled_fa_gb300 import inputs
    f = (rng.standard_normal(n) * scale).astype(np.float32)
    return inputs.bf16_bits_to_f32(inputs.f32_to_bf16_bits(f)).astype(np.float64)


def test_block_properties_random():
    rng = np.random.default_rng(7)
    x = _bf16_exact(rng, 64 * 32).reshape(64, 32)
    x[3] *= 1e-3
    x[7] *= 300.0
    q, s = oracle.quantize(x, oracle.ROW)
    deq = oracle.dequantize(q, s, oracle.ROW)
    # power-of-two equivariance: scaling a block by 2^k shifts only the scale
    for k in (-5, 1, 9):
        q2, s2 = oracle.quantize(x * 2.0 ** k, oracle.ROW)
        np.testing.assert_array_equal(q2, q)
        np.testing.assert_array_equal(s2.astype(int), s.astype(int) + k)
    # sign symmetry: negation flips only the payload sign bit
    q3, s3 = oracle.quantize(-x, oracle.ROW)
    np.testing.assert_array_equal(s3, s)
    np.testing.assert_array_equal(q3, q ^ 0x80)
    # idempotence on dequantized values
    q4, s4 = oracle.quantize(deq, oracle.ROW)
    np.testing.assert_array_equal(q4, q)
    np.testing.assert_array_equal(s4, s)
    # error bound: half a quantum of the scaled value's binade
    X = s.astype(int) - 127
    scaled = x * 2.0 ** (-X[:, :1])
    err = np.abs(deq - x) * 2.0 ** (-X[:, :1])
    e = np.floor(np.log2(np.maximum(np.abs(scaled), 2.0 ** -6)))
    bound = 2.0 ** (e - 4)
    sat = np.abs(scaled) > 448
    assert np.all(err[~sat] <= bound[~sat] * (1 + 1e-12))
    # the block maximum lands in [256, 512) -> payload magnitude 256..448
    amax_code = np.max(q & 0x7F, axis=1)
    assert np.all(amax_code >= 0x78)
