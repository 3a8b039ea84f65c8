"""GPU MXFP4 / MXFP6 / NVFP4 quantizers and the GEMM on MXFP6 / MXFP4 operands
vs the CPU oracle: codes, scales and the NVFP4 tensor scale bit-exact; the
GEMM bit-exact where its fp32 accumulation is exact."""
import numpy as np
import pytest

import oracle
from mxfp8_block_scaled_fa_gb300 import inputs
from tests.helpers import host, to_dev, unpack_packed

pytestmark = pytest.mark.gpu

FMTS = [(0, oracle.E2M1), (1, oracle.E2M3), (2, oracle.E3M2)]   # (library, oracle) codes


@pytest.fixture(scope="module")
def mx():
    import torch
    from mxfp8_block_scaled_fa_gb300 import build, mxfa
    build.build()
    assert torch.cuda.is_available()
    return mxfa


def _special_rows(cols, rng):
    """Blocks at the rule's edges: powers of two, ties, tiny, huge, Inf, NaN."""
    x = rng.standard_normal((8, cols)).astype(np.float32)
    x[0, :32] = 6.0
    x[1, :32] = np.linspace(-7.5, 7.5, 32)
    x[2, :32] = 2.0 ** -130                 # bf16 subnormals: scale clamped at 0
    x[3, :32] = 3.0e38
    x[4, 5] = np.inf
    x[5, 7] = np.nan
    x[6, :32] = [0.25, 0.75, 2.5, 5.0] * 8  # E2M1 ties with scale 2^0
    x[7, :32] = 28.0
    return x


def _mma_form(codes, bits):
    """One code per byte -> the MMA operand form: each run of 16 codes packed
    little-endian (`bits` bits each) at the start of a 16-byte group, rest zero."""
    rows, cols = codes.shape
    g = codes.reshape(rows, cols // 16, 16).astype(np.uint64)
    out = np.zeros((rows, cols // 16, 16), np.uint8)
    for j in range(16):                       # code j -> bits [bits*j, bits*j + bits)
        for b in range(bits):
            pos = bits * j + b
            out[:, :, pos // 8] |= (((g[:, :, j] >> np.uint64(b)) & np.uint64(1)) << np.uint64(pos % 8)).astype(np.uint8)
    return out.reshape(rows, cols)


@pytest.mark.parametrize("lib_fmt,o_fmt", FMTS)
def test_mx_lowp_quantize(mx, lib_fmt, o_fmt):
    import torch
    rng = np.random.default_rng(40 + lib_fmt)
    x = np.concatenate([rng.standard_normal((248, 512)).astype(np.float32) * 3, _special_rows(512, rng)])
    bits = inputs.f32_to_bf16_bits(x)
    res = mx.quantize_lowp(to_dev(bits), lib_fmt, packed=True)
    res_mma = mx.quantize_lowp(to_dev(bits), lib_fmt, mma=True)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    q_ref, s_ref = oracle.quantize_mx(inputs.bf16_bits_to_f32(bits).astype(np.float64), o_fmt)
    np.testing.assert_array_equal(host(res["sf"]), s_ref)
    np.testing.assert_array_equal(host(res["q"]), q_ref)
    np.testing.assert_array_equal(host(res_mma["sf"]), s_ref)
    np.testing.assert_array_equal(host(res_mma["q"]), _mma_form(q_ref, 4 if lib_fmt == 0 else 6))
    # packed atoms (the GEMM's layout) decode to the compact scales
    comp, _ = unpack_packed(host(res["sf_packed"]), 0, [256], 512 // 128)
    np.testing.assert_array_equal(comp, s_ref)


def test_mma_form_helper():
    # the test's own repacking, on a hand-worked run: FP4 codes 1..15,0 give
    # nibbles 0x21, 0x43, ...; FP6 codes 1, 2 give 0b000010_000001 = 0x81, 0x00
    c = np.zeros((1, 16), np.uint8)
    c[0] = list(range(1, 16)) + [0]
    assert _mma_form(c, 4)[0, :8].tolist() == [0x21, 0x43, 0x65, 0x87, 0xA9, 0xCB, 0xED, 0x0F]
    assert not _mma_form(c, 4)[0, 8:].any()
    c6 = np.zeros((1, 16), np.uint8)
    c6[0, :2] = [1, 2]
    c6[0, 15] = 0x3F
    f = _mma_form(c6, 6)[0]
    assert f[:2].tolist() == [0x81, 0x00] and f[11] == 0xFC and not f[12:].any()


def test_nvfp4_quantize(mx):
    import torch
    rng = np.random.default_rng(50)
    x = rng.standard_normal((256, 512)).astype(np.float32) * 5
    x[3, :16] = 0.0
    x[7, 20] = 900.0
    bits = inputs.f32_to_bf16_bits(x)
    res = mx.quantize_lowp(to_dev(bits), mx.LOWP_NVFP4)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    q_ref, s_ref, st = oracle.quantize_nvfp4(inputs.bf16_bits_to_f32(bits).astype(np.float64))
    assert host(res["tensor_scale"])[0] == np.float32(st)
    np.testing.assert_array_equal(host(res["sf"]), s_ref)
    np.testing.assert_array_equal(host(res["q"]), q_ref)


VALUES = {0: [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0],          # E2M1 magnitudes
          1: [0.0, 0.25, 0.5, 1.0, 1.25, 2.0, 3.5, 7.5],       # E2M3
          2: [0.0, 0.25, 1.0, 1.5, 3.0, 4.0, 12.0, 28.0]}      # E3M2


@pytest.mark.parametrize("a_fmt,b_fmt", [(0, 0), (1, 1), (2, 2), (0, None), (2, 1)])
def test_gemm_on_lowp_operands_exact(mx, a_fmt, b_fmt):
    # operands drawn from values every block scale keeps exact, small enough
    # that the fp32 accumulation is exact: Y, its bf16 copy and its MXFP8
    # quantization equal the oracle's bit for bit
    import torch
    M, N, K = 256, 256, 512
    rng = np.random.default_rng(60 + a_fmt)

    def operand(rows, fmt):
        if fmt is None:   # MXFP8 (E4M3) operand: small integers
            v = rng.integers(-8, 9, size=(rows, K)).astype(np.float32)
            m = mx.quantize(to_dev(inputs.f32_to_bf16_bits(v).reshape(rows, K // 128, 128)), mx.ROW,
                            mx.Seqs.dense(1, rows))
            return v, m.mx_in(), mx.ELEM_E4M3
        v = (rng.choice(VALUES[fmt], size=(rows, K)) * rng.choice([-1.0, 1.0], size=(rows, K))).astype(np.float32)
        r = mx.quantize_lowp(to_dev(inputs.f32_to_bf16_bits(v)), fmt, packed=True, mma=True)
        o_fmt = dict(FMTS)[fmt]
        q_ref, s_ref = oracle.quantize_mx(v.astype(np.float64), o_fmt)
        np.testing.assert_array_equal(oracle.dequantize_mx(q_ref, s_ref, o_fmt), v)   # exact operand
        np.testing.assert_array_equal(host(r["q"]), _mma_form(q_ref, 4 if fmt == 0 else 6))
        keep.append(r)
        return v, mx.MxIn(r["q"].data_ptr(), r["sf_packed"].data_ptr()), [mx.ELEM_E2M1, mx.ELEM_E2M3,
                                                                           mx.ELEM_E3M2][fmt]
    keep = []
    a, a_in, af = operand(M, a_fmt)
    b, b_in, bf = operand(N, b_fmt)
    u8 = dict(dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    row = [torch.empty((M, N), **u8), torch.empty((M, N // 32), **u8), torch.empty(M // 128 * N // 128 * 512, **u8)]
    out_row = mx.MxOut(*(t.data_ptr() for t in row))
    mx.mxfa_gemm_quant_fmt(a_in, af, b_in, bf, M, N, K, y, out_row, None)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    yref = a.astype(np.float64) @ b.astype(np.float64).T
    np.testing.assert_array_equal(oracle.gemm_nt(a, b), yref)
    np.testing.assert_array_equal(host(y.view(torch.int16)).view(np.uint16),
                                  inputs.f32_to_bf16_bits(yref.astype(np.float32)))
    q_ref, s_ref = oracle.quantize(yref, oracle.ROW)
    np.testing.assert_array_equal(host(row[0]), q_ref)
    np.testing.assert_array_equal(host(row[1]), s_ref)
