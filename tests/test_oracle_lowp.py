"""The oracle's lower-precision formats (MXFP4 = E2M1, MXFP6 = E2M3 / E3M2 with
E8M0 scales per 32; NVFP4 = E2M1 with E4M3 scales per 16 and an fp32 tensor
scale), pinned by the OCP format definitions, hand-worked blocks and
invariants (CPU only)."""
import numpy as np
import pytest

import oracle

E2M1, E2M3, E3M2 = oracle.E2M1, oracle.E2M3, oracle.E3M2


def test_e2m1_code_table():
    # sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent 0 is
    # subnormal (m * 2^-1): the eight magnitudes of FP4
    np.testing.assert_array_equal(oracle.fp_decode(E2M1, range(8)),
                                  [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    np.testing.assert_array_equal(oracle.fp_decode(E2M1, range(8, 16)),
                                  -np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]))


@pytest.mark.parametrize("fmt,maxv,min_sub,ncodes", [(E2M1, 6.0, 0.5, 16), (E2M3, 7.5, 0.125, 64),
                                                     (E3M2, 28.0, 0.0625, 64)])
def test_format_closed_forms(fmt, maxv, min_sub, ncodes):
    assert oracle.fp_max(fmt) == maxv
    vals = oracle.fp_decode(fmt, range(ncodes // 2))
    assert vals[1] == min_sub
    assert np.all(np.diff(vals) > 0)                  # codes ordered by value
    # every value encodes to its own code (round trip), both signs
    codes = np.arange(ncodes, dtype=np.uint8)
    back = oracle.fp_encode(fmt, oracle.fp_decode(fmt, codes))
    pos_zero, neg_zero = 0, ncodes // 2
    expect = codes.copy()
    np.testing.assert_array_equal(back[codes != neg_zero], expect[codes != neg_zero])


def test_e2m1_rounding_ties_and_saturation():
    # ties go to the even code: 0.25 -> 0, 0.75 -> 1.0, 2.5 -> 2.0, 5.0 -> 4.0
    got = oracle.fp_decode(E2M1, oracle.fp_encode(E2M1, [0.25, 0.75, 2.5, 5.0, 100.0, -5.0, 1.26]))
    np.testing.assert_array_equal(got, [0.0, 1.0, 2.0, 4.0, 6.0, -4.0, 1.5])


def test_mxfp4_blocks_hand_worked():
    x = np.zeros((3, 32))
    x[0, :] = 1.0; x[0, 0] = 6.0          # amax 6: floor(log2 6) - 2 = 0 -> scale 127
    x[1, :] = 1.0; x[1, 0] = 12.0         # amax 12: exponent 3 - 2 = 1 -> 128; 12/2 = 6, 1/2 = 0.5
    x[2, 0] = 2.0 ** -140                 # tiny block: clamped at scale 0
    q, s = oracle.quantize_mx(x, E2M1)
    np.testing.assert_array_equal(s[:, 0], [127, 128, 0])
    assert q[0, 0] == 7 and np.all(q[0, 1:] == 2)
    assert q[1, 0] == 7 and np.all(q[1, 1:] == 1)
    # 2^-140 * 2^127 = 2^-13: far below half of the smallest step 0.5 -> 0
    assert q[2, 0] == 0


def test_mxfp6_blocks_hand_worked():
    x = np.zeros((2, 32))
    x[0, 0], x[0, 1] = 28.0, 0.0625       # E3M2: amax 28, exponent 4 - 4 = 0; 0.0625 = min subnormal
    x[1, 0], x[1, 1] = 7.5, 0.125         # E2M3: amax 7.5, exponent 2 - 2 = 0; 0.125 = min subnormal
    q3, s3 = oracle.quantize_mx(x[:1], E3M2)
    q2, s2 = oracle.quantize_mx(x[1:], E2M3)
    assert s3[0, 0] == 127 and oracle.fp_decode(E3M2, [q3[0, 0], q3[0, 1]]).tolist() == [28.0, 0.0625]
    assert s2[0, 0] == 127 and oracle.fp_decode(E2M3, [q2[0, 0], q2[0, 1]]).tolist() == [7.5, 0.125]


@pytest.mark.parametrize("fmt", [E2M1, E2M3, E3M2])
def test_mx_scale_equivariance_and_error_bound(fmt):
    # scaling by 2^k keeps the codes and adds k to the scale (away from the
    # clamps); each dequantized value lies within half a step of its input
    # (or at the block's saturation value)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((8, 64))
    q, s = oracle.quantize_mx(x, fmt)
    q2, s2 = oracle.quantize_mx(x * 2.0 ** 5, fmt)
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(s2.astype(int), s.astype(int) + 5)
    y = oracle.dequantize_mx(q, s, fmt)
    mb = {E2M1: 1, E2M3: 3, E3M2: 2}[fmt]
    step = np.abs(y) * 2.0 ** -mb + np.ldexp(1.0, np.repeat(s.astype(np.int64), 32, axis=1) - 127)
    assert np.all(np.abs(y - x) <= step)


def test_nvfp4_hand_worked():
    # block 0: amax 2688 = 448 * 6 makes the tensor scale 1; its E4M3 scale is
    # 2688 / 6 = 448 (0x7E) and 2688 / 448 = 6 (code 7), 1 / 448 -> 0.
    # block 1: amax 3 -> scale 3 / 6 = 0.5 (E4M3 0x30): 3 -> 6 (7), 1.5 -> 3 (5),
    # 0.75 -> 1.5 (3)
    x = np.zeros((1, 32))
    x[0, 0], x[0, 1] = 2688.0, 1.0
    x[0, 16], x[0, 17], x[0, 18] = 3.0, 1.5, 0.75
    q, s, st = oracle.quantize_nvfp4(x)
    assert st == 1.0
    assert s[0, 0] == 0x7E and s[0, 1] == 0x30
    assert q[0, 0] == 7 and q[0, 1] == 0
    assert (q[0, 16], q[0, 17], q[0, 18]) == (7, 5, 3)
    assert np.all(q[0, 19:] == 0)
