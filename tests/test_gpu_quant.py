"""GPU quantizers and fused RMSNorm+Quantize vs the CPU oracle: bit-exact
payload bytes and E8M0 scales (compact, and packed after decoding)."""
import numpy as np
import pytest

import oracle
from mxfp8_block_scaled_fa_gb300 import inputs
from tests.helpers import f64, host, to_dev, unpack_packed

pytestmark = pytest.mark.gpu

MODES = [(0, "row"), (1, "col"), (2, "sq")]


@pytest.fixture(scope="module")
def mx():
    import torch
    from mxfp8_block_scaled_fa_gb300 import build, mxfa
    build.build()
    assert torch.cuda.is_available()
    return mxfa


def _check_quant(mx, bits3, lens, H, blk):
    import torch
    tokens = bits3.shape[0]
    if lens is None:
        seqs = mx.Seqs.dense(1, tokens)
        lens_ = [tokens]
        cu = None
    else:
        seqs = mx.Seqs.varlen(lens, "cuda")
        lens_ = lens
        cu = seqs.cu_host
    m = mx.quantize(to_dev(bits3), blk, seqs)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    q_ref, s_ref = oracle.quantize(f64(bits3).reshape(tokens, -1), blk, cu)
    np.testing.assert_array_equal(host(m.data).reshape(tokens, -1), q_ref)
    np.testing.assert_array_equal(host(m.sf_compact), s_ref)
    comp, pad = unpack_packed(host(m.sf_packed), blk, lens_, H)
    np.testing.assert_array_equal(comp, s_ref)
    assert np.all(pad == 0x7F)
    packed2 = mx.sf_pack(m.sf_compact, blk, seqs, H)
    # the C-ABI round trip of the packed layout: unpack gives the compact scales back
    comp2 = mx.sf_unpack(m.sf_packed, blk, seqs, H)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    np.testing.assert_array_equal(host(packed2), host(m.sf_packed))
    np.testing.assert_array_equal(host(comp2), s_ref)


def _check_dual(mx, bits3, lens, H, blk):
    # one read, two layouts: blk (COL or SQ) and ROW, each equal to the
    # oracle's quantization of the same bf16 tensor, compact and packed
    import torch
    tokens = bits3.shape[0]
    seqs = mx.Seqs.varlen(lens, "cuda") if lens is not None else mx.Seqs.dense(1, tokens)
    lens_ = lens if lens is not None else [tokens]
    cu = seqs.cu_host
    first, row = mx.quantize_dual(to_dev(bits3), blk, seqs)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for m, b in ((first, blk), (row, mx.ROW)):
        q_ref, s_ref = oracle.quantize(f64(bits3).reshape(tokens, -1), b, cu)
        np.testing.assert_array_equal(host(m.data).reshape(tokens, -1), q_ref, err_msg=str(b))
        np.testing.assert_array_equal(host(m.sf_compact), s_ref, err_msg=str(b))
        comp, pad = unpack_packed(host(m.sf_packed), b, lens_, H)
        np.testing.assert_array_equal(comp, s_ref, err_msg=str(b))
        assert np.all(pad == 0x7F), b


@pytest.mark.parametrize("blk", [1, 2])
@pytest.mark.parametrize("case", ["dense", "ragged", "empty", "odd_heads"])
def test_quantize_dual(mx, blk, case):
    if case == "dense":
        q, _, _, _ = inputs.dense_attn(2, 2, 384, 128, seed=7)
        _check_dual(mx, q.reshape(768, 2, 128), None, 2, blk)
    elif case == "ragged":
        lens = [5, 130, 64, 33, 1, 257]
        q, _, _, _, _, _ = inputs.varlen_attn(lens, lens, 3, 128, seed=8)
        _check_dual(mx, q, lens, 3, blk)
    elif case == "empty":
        lens = [0, 40, 0, 129, 0]
        q, _, _, _, _, _ = inputs.varlen_attn(lens, lens, 2, 128, seed=9)
        _check_dual(mx, q, lens, 2, blk)
    else:  # 5 heads: the last warp of a column block is partly idle
        q, _, _, _ = inputs.dense_attn(1, 5, 160, 128, seed=10, outliers=True)
        _check_dual(mx, q.reshape(160, 5, 128), None, 5, blk)


@pytest.mark.parametrize("B,S,H", [(3, 200, 3), (2, 96, 4), (4, 128, 1), (3, 5, 2)])
def test_quantize_dense_batches(mx, B, S, H):
    # dense batches of several sequences whose length is not a multiple of the
    # 128-row tile (padding blocks inside each sequence's last tile), odd head
    # counts (a half-used column chunk), a tensor shorter than one 32-row
    # block: every kind, single and dual output
    import torch
    q, _, _, _ = inputs.dense_attn(B, H, S, 128, seed=12 + S)
    bits3 = q.reshape(B * S, H, 128)
    tokens = B * S
    seqs = mx.Seqs.dense(B, S)
    lens = [S] * B
    cu = np.arange(B + 1, dtype=np.int32) * S
    x64 = f64(bits3).reshape(tokens, -1)
    ref = {b: oracle.quantize(x64, b, cu) for b in (0, 1, 2)}

    def check(m, b):
        q_ref, s_ref = ref[b]
        np.testing.assert_array_equal(host(m.data).reshape(tokens, -1), q_ref, err_msg=str(b))
        np.testing.assert_array_equal(host(m.sf_compact), s_ref, err_msg=str(b))
        comp, pad = unpack_packed(host(m.sf_packed), b, lens, H)
        np.testing.assert_array_equal(comp, s_ref, err_msg=str(b))
        assert np.all(pad == 0x7F), b

    dev = to_dev(bits3)
    for b in (0, 1, 2):
        m = mx.quantize(dev, b, seqs)
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        check(m, b)
    for b in (1, 2):
        first, row = mx.quantize_dual(dev, b, seqs)
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        check(first, b)
        check(row, 0)


@pytest.mark.parametrize("blk,name", MODES)
def test_quantize_tiny_dense(mx, blk, name):
    q, _, _, _ = inputs.dense_attn(1, 2, 256, 128, seed=0)
    _check_quant(mx, q.reshape(256, 2, 128), None, 2, blk)


@pytest.mark.parametrize("blk,name", MODES)
def test_quantize_ragged_varlen(mx, blk, name):
    lens = [5, 130, 64, 33, 1, 257]
    q, _, _, _, _, _ = inputs.varlen_attn(lens, lens, 3, 128, seed=5)
    _check_quant(mx, q, lens, 3, blk)


@pytest.mark.parametrize("blk,name", MODES)
def test_quantize_varlen_with_empty_sequences(mx, blk, name):
    # zero-length sequences own no payload row, no scale row and no packed tile
    lens = [0, 40, 0, 0, 129, 0]
    q, _, _, _, _, _ = inputs.varlen_attn(lens, lens, 2, 128, seed=6)
    _check_quant(mx, q, lens, 2, blk)


@pytest.mark.parametrize("blk,name", MODES)
def test_quantize_adversarial_blocks(mx, blk, name):
    # zeros, -0, the 448 boundary, E4M3 subnormals, ties, huge / tiny values,
    # and Inf / NaN blocks, laid out so every block kind meets them
    rng = np.random.default_rng(11)
    x = rng.standard_normal((128, 2, 128)).astype(np.float32)
    flat = x.reshape(128, 256)
    flat[0:32, 0:32] = 0.0
    flat[1, 5] = -0.0
    flat[32:64, 32:64] = 1.0
    flat[40, 40] = 1.75
    flat[41, 41] = 1.875
    flat[64, 64:96] = [1.0] + [2.0 ** -17, 2.0 ** -18, 1.5 * 2 ** -17, 3 * 2 ** -19] + [0.0] * 27
    flat[65, 64:68] = [1.0, 17 * 2.0 ** -9, 19 * 2.0 ** -9, 31 * 2.0 ** -9]
    flat[96:128, 96:128] *= 2.0 ** 120
    flat[70, 130] = 1.9921875 * 2.0 ** 127
    flat[71, 131] = 2.0 ** -130
    flat[100, 200] = np.inf
    flat[101, 210] = -np.inf
    flat[102, 220] = np.nan
    bits = inputs.f32_to_bf16_bits(x)
    _check_quant(mx, bits, None, 2, blk)


def test_quantize_full_llm_tensor(mx):
    # one full Q tensor of the LLM-shaped workload (B2 S8192 H16), all kinds
    import torch
    B, S, H, D = 2, 8192, 16, 128
    q = inputs.normal_bf16((B, S, H, D), 1)
    dev = to_dev(q)
    seqs = mx.Seqs.dense(B, S)
    x64 = f64(q).reshape(B * S, H * D)
    cu = np.array([0, S, 2 * S], np.int32)
    refs = {}
    for blk in (0, 1, 2):
        m = mx.quantize(dev, blk, seqs)
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        q_ref, s_ref = oracle.quantize(x64, blk, cu)
        np.testing.assert_array_equal(host(m.data).reshape(B * S, -1), q_ref)
        np.testing.assert_array_equal(host(m.sf_compact), s_ref)
        refs[blk] = (q_ref, s_ref)
    # the one-read dual outputs, as the training step uses them
    for blk in (1, 2):
        first, row = mx.quantize_dual(dev, blk, seqs)
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        for m, b in ((first, blk), (row, 0)):
            np.testing.assert_array_equal(host(m.data).reshape(B * S, -1), refs[b][0], err_msg=str(b))
            np.testing.assert_array_equal(host(m.sf_compact), refs[b][1], err_msg=str(b))


@pytest.mark.parametrize("T,C,H,seg", [(256, 2048, 16, 128), (96, 256, 2, 32), (384, 512, 4, 128)])
def test_rmsnorm_quant_small(mx, T, C, H, seg):
    import torch
    x = inputs.normal_bf16((T, C), 7)
    g = np.random.default_rng(8).uniform(0.5, 1.5, C).astype(np.float32)
    packed = (T % seg == 0) and (seg % 128 == 0)
    res = mx.rmsnorm_quant(to_dev(x), torch.from_numpy(g).cuda(), 1e-6, seg, H, packed=packed)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    ref = oracle.rmsnorm_quant(inputs.bf16_bits_to_f32(x), g, 1e-6, 7, seg)
    for name, blk in (("row", 0), ("col", 1), ("sq", 2)):
        np.testing.assert_array_equal(host(res[name].data), ref[name][0], err_msg=name)
        np.testing.assert_array_equal(host(res[name].sf_compact), ref[name][1], err_msg=name)
        if packed:
            comp, pad = unpack_packed(host(res[name].sf_packed), blk, [seg] * (T // seg), H)
            np.testing.assert_array_equal(comp, ref[name][1], err_msg=name)


def test_rmsnorm_quant_full_fused_config(mx):
    # the fused producer workload: X [32768, 2048], gamma U[0.5, 1.5], eps 1e-6
    import torch
    x, g, _ = inputs.fused_inputs()
    res = mx.rmsnorm_quant(to_dev(x), torch.from_numpy(g).cuda(), 1e-6, 8192, 16)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    ref = oracle.rmsnorm_quant(inputs.bf16_bits_to_f32(x), g, 1e-6, 7, 8192)
    for name in ("row", "col", "sq"):
        np.testing.assert_array_equal(host(res[name].data), ref[name][0], err_msg=name)
        np.testing.assert_array_equal(host(res[name].sf_compact), ref[name][1], err_msg=name)


def test_rmsnorm_quant_inf_nan_rows(mx):
    # an Inf and a NaN in the input: their rows normalise to NaN / 0 values,
    # so row, column and square blocks holding them take scale 0xFF and 0x7F
    # payloads, exactly as the oracle's OCP rule says
    import torch
    T, C, H, seg = 96, 256, 2, 32
    x = inputs.normal_bf16((T, C), 9)
    x[5, 10] = 0x7F80   # +Inf (bf16 bits)
    x[40, 100] = 0x7FC0  # NaN
    g = np.random.default_rng(10).uniform(0.5, 1.5, C).astype(np.float32)
    res = mx.rmsnorm_quant(to_dev(x), torch.from_numpy(g).cuda(), 1e-6, seg, H, packed=False)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    ref = oracle.rmsnorm_quant(inputs.bf16_bits_to_f32(x), g, 1e-6, 7, seg)
    assert (ref["col"][1] == 0xFF).any() and (ref["row"][1] == 0xFF).any()
    for name in ("row", "col", "sq"):
        np.testing.assert_array_equal(host(res[name].data), ref[name][0], err_msg=name)
        np.testing.assert_array_equal(host(res[name].sf_compact), ref[name][1], err_msg=name)
