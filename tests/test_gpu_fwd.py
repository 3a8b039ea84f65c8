"""GPU forward (tcgen05 kernel) vs the CPU oracle on the same seeded inputs.

Bar: O relative Frobenius <= 1e-2 and max-abs <= 3e-2; LSE max-abs <= 1e-4;
each max-abs bar plus the rounding of the output format (bf16 O, fp32 lse).
The oracle is the method's fp64 definition over the dequantized MXFP8
operands, with the kernel's declared schedule: 128-key tiles in ascending
order, running max moved when it grows by more than 8 (log2 units).
"""
import math

import numpy as np
import pytest

import oracle
from mxfp8_block_scaled_fa_gb300 import inputs
from tests.helpers import f64, host, max_abs, rel_fro, to_dev

pytestmark = pytest.mark.gpu

THR = 8.0
O_REL, O_ABS, LSE_ABS = 1e-2, 3e-2, 1e-4


@pytest.fixture(scope="module")
def mx():
    import torch
    from mxfp8_block_scaled_fa_gb300 import build, mxfa
    build.build()
    assert torch.cuda.is_available()
    return mxfa


def gpu_fwd(mx, qb, kb, vb, seqs_q, seqs_k, scale, causal):
    import torch
    q = mx.quantize(to_dev(qb), mx.ROW, seqs_q)
    k = mx.quantize(to_dev(kb), mx.ROW, seqs_k)
    v = mx.quantize(to_dev(vb), mx.COL, seqs_k)
    o, lse = mx.attention_fwd(q, k, v, seqs_q, seqs_k, scale, causal)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    return host(o.float()).astype(np.float64), host(lse)


def _spacing(x, mant_bits):
    """Distance between adjacent numbers near |x| in a format with mant_bits."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - mant_bits)


def check(o, lse, oo, lo):
    # O is returned in bf16 and lse in fp32: the max-abs bars add the output
    # format's own rounding (half a bf16 spacing of O, four fp32 spacings of
    # lse), which only matters where |O| > 8 or |lse| > 100
    print(f"[fwd parity] O rel-Fro {rel_fro(o, oo):.3e} max-abs {max_abs(o, oo):.3e} "
          f"lse max-abs {max_abs(lse, lo):.3e}")
    assert rel_fro(o, oo) <= O_REL, rel_fro(o, oo)
    excess = np.abs(o - oo) - 0.5 * _spacing(oo, 7)
    assert excess.max() <= O_ABS, (max_abs(o, oo), excess.max())
    lexcess = np.abs(lse - lo) - 4 * _spacing(lo, 23)
    assert lexcess.max() <= LSE_ABS, (max_abs(lse, lo), lexcess.max())


@pytest.mark.parametrize("B,H,S,causal", [
    (1, 2, 256, False),     # the tiny workload
    (1, 2, 384, True),
    (2, 3, 300, False),     # ragged tail inside a 128-key tile
    (2, 2, 300, True),
    (1, 1, 1, False),       # single key
    (1, 2, 33, True),
    (3, 2, 640, True),      # several tiles per head, more than the K/V ring
    (4, 20, 1000, True),    # more work items than SMs: a CTA walks several items
    (2, 40, 768, False),
])
def test_fwd_dense(mx, B, H, S, causal):
    D = 128
    scale = 1 / math.sqrt(D)
    qb, kb, vb, _ = inputs.dense_attn(B, H, S, D, seed=100 + S)
    seqs = mx.Seqs.dense(B, S)
    o, lse = gpu_fwd(mx, qb, kb, vb, seqs, seqs, scale, causal)
    cu = np.arange(0, (B + 1) * S, S, dtype=np.int32)
    f = lambda b: f64(b).reshape(B * S, H, D)
    oo, lo = oracle.method_fwd(f(qb), f(kb), f(vb), cu, cu, scale, causal, True, 128, THR)
    check(o.reshape(B * S, H, D), lse.reshape(B, H, S).transpose(1, 0, 2).reshape(H, B * S), oo, lo)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_varlen(mx, causal):
    H, D = 2, 128
    lq = [64, 300, 7, 129, 1, 255]
    lk = lq if causal else [32, 200, 1, 260, 77, 128]
    qb, kb, vb, _, cu_q, cu_k = inputs.varlen_attn(lq, lk, H, D, seed=21)
    sq = mx.Seqs.varlen(lq, "cuda")
    sk = mx.Seqs.varlen(lk, "cuda")
    scale = 1 / math.sqrt(D)
    o, lse = gpu_fwd(mx, qb, kb, vb, sq, sk, scale, causal)
    oo, lo = oracle.method_fwd(f64(qb), f64(kb), f64(vb), cu_q, cu_k, scale, causal, True, 128, THR)
    check(o, lse, oo, lo)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_varlen_empty_sequences(mx, causal):
    # zero-length query and key sequences: a query whose key sequence is empty
    # gets O = 0 and lse = -inf; an empty query sequence writes nothing
    H, D = 2, 128
    lq = [0, 70, 5, 0, 130]
    lk = [0, 70, 0, 9, 130] if not causal else [0, 70, 0, 0, 130]
    qb, kb, vb, _, cu_q, cu_k = inputs.varlen_attn(lq, lk, H, D, seed=23)
    sq = mx.Seqs.varlen(lq, "cuda")
    sk = mx.Seqs.varlen(lk, "cuda")
    scale = 1 / math.sqrt(D)
    o, lse = gpu_fwd(mx, qb, kb, vb, sq, sk, scale, causal)
    oo, lo = oracle.method_fwd(f64(qb), f64(kb), f64(vb), cu_q, cu_k, scale, causal, True, 128, THR)
    empty = np.repeat(np.asarray(lk) == 0, lq)       # query tokens with no key
    assert empty.sum() == 5
    assert np.all(o[empty] == 0) and np.all(oo[empty] == 0)
    assert np.all(np.isneginf(lse[:, empty])) and np.all(np.isneginf(lo[:, empty]))
    check(o[~empty], lse[:, ~empty], oo[~empty], lo[:, ~empty])


@pytest.mark.parametrize("thr,p_scale,varlen", [
    (0.0, 0, False),   # exact rescale at every increase of the running max
    (4.0, 0, True),
    (8.0, 1, False),   # constant P scale with the default threshold
    (0.0, 1, True),
    (2.5, 1, False),   # a non-integer threshold: constant exponent ceil(2.5) - 8
])
def test_fwd_options(mx, thr, p_scale, varlen):
    # the rescale threshold and the P scale mode against the oracle run with
    # the same options
    H, D = 2, 128
    scale = 1 / math.sqrt(D)
    if varlen:
        lens = [64, 300, 7, 129, 1, 255]
        qb, kb, vb, _, cu, _ = inputs.varlen_attn(lens, lens, H, D, seed=61)
        seqs = mx.Seqs.varlen(lens, "cuda")
    else:
        B, S = 2, 384
        qb, kb, vb, _ = (b.reshape(B * S, H, D) for b in inputs.dense_attn(B, H, S, D, seed=62))
        cu = np.arange(0, (B + 1) * S, S, dtype=np.int32)
        seqs = mx.Seqs.dense(B, S)
    import torch
    opts = mx.AttnOpts(thr, p_scale)
    q = mx.quantize(to_dev(qb), mx.ROW, seqs)
    k = mx.quantize(to_dev(kb), mx.ROW, seqs)
    v = mx.quantize(to_dev(vb), mx.COL, seqs)
    o, lse = mx.attention_fwd(q, k, v, seqs, seqs, scale, True, opts=opts)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    oo, lo = oracle.method_fwd(f64(qb), f64(kb), f64(vb), cu, cu, scale, True, True, 128, thr,
                               p_scale)
    og = host(o.float()).astype(np.float64)
    lg = host(lse)
    if not varlen:
        lg = lg.reshape(2, H, 384).transpose(1, 0, 2).reshape(H, -1)
    check(og, lg, oo, lo)


@pytest.mark.parametrize("outliers_v", [False, True])
def test_fwd_outliers_small(mx, outliers_v):
    # the outlier recipe (1% of Q/K channels x20, 0.1% of elements x200);
    # outliers_v also puts 0.1% x200 elements into V (non-uniform V scales)
    B, H, S, D = 1, 4, 512, 128
    qb, kb, vb, _ = inputs.dense_attn(B, H, S, D, seed=2, outliers=True, outliers_v=outliers_v)
    seqs = mx.Seqs.dense(B, S)
    scale = 1 / math.sqrt(D)
    o, lse = gpu_fwd(mx, qb, kb, vb, seqs, seqs, scale, False)
    f = lambda b: f64(b).reshape(B * S, H, D)
    oo, lo = oracle.method_fwd(f(qb), f(kb), f(vb), None, None, scale, False, True, 128, THR)
    check(o.reshape(B * S, H, D), lse.reshape(H, S), oo, lo)


def test_fwd_llm_config_sampled_heads(mx):
    # full LLM-shaped causal workload on the GPU, as the benchmark launches it;
    # the oracle recomputes two sampled (batch, head) pairs in full
    B, H, S, D = 2, 16, 8192, 128
    scale = 1 / math.sqrt(D)
    qb, kb, vb, _ = inputs.dense_attn(B, H, S, D, seed=1)
    seqs = mx.Seqs.dense(B, S)
    o, lse = gpu_fwd(mx, qb, kb, vb, seqs, seqs, scale, True)
    o = o.reshape(B, S, H, D)
    lse = lse.reshape(B, H, S)
    for b, h in ((0, 3), (1, 14)):
        sl = lambda x: f64(x[b, :, h:h + 1, :])
        oo, lo = oracle.method_fwd(sl(qb), sl(kb), sl(vb), None, None, scale, True, True, 128, THR)
        check(o[b, :, h:h + 1, :], lse[b, h:h + 1, :], oo, lo)


@pytest.mark.parametrize("varlen", [False, True])
def test_fwd_mxfp8_output(mx, varlen):
    # the forward that also emits O as MXFP8 (1x32 blocks along D): its bf16 O
    # equals the plain forward's bit for bit, and its payload and scales equal
    # the oracle's ROW quantization of that bf16 O, byte for byte
    import torch
    from tests.helpers import unpack_packed
    H, D = 2, 128
    if varlen:
        lens = [64, 300, 7, 129, 1, 255]
        qb, kb, vb, _, cu, _ = inputs.varlen_attn(lens, lens, H, D, seed=41)
        seqs = mx.Seqs.varlen(lens, "cuda")
    else:
        B, S = 2, 300
        lens = [S] * B
        qb, kb, vb, _ = inputs.dense_attn(B, H, S, D, seed=42)
        qb, kb, vb = (b.reshape(B * S, H, D) for b in (qb, kb, vb))
        cu = np.arange(0, (B + 1) * S, S, dtype=np.int32)
        seqs = mx.Seqs.dense(B, S)
    scale = 1 / math.sqrt(D)
    q = mx.quantize(to_dev(qb), mx.ROW, seqs)
    k = mx.quantize(to_dev(kb), mx.ROW, seqs)
    v = mx.quantize(to_dev(vb), mx.COL, seqs)
    o_plain, lse_plain = mx.attention_fwd(q, k, v, seqs, seqs, scale, True)
    o, lse, omx = mx.attention_fwd(q, k, v, seqs, seqs, scale, True, o_mx=True)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    o_bits = host(o.view(torch.int16)).view(np.uint16)
    np.testing.assert_array_equal(o_bits, host(o_plain.view(torch.int16)).view(np.uint16))
    np.testing.assert_array_equal(host(lse), host(lse_plain))
    tokens = o_bits.shape[0]
    q_ref, s_ref = oracle.quantize(f64(o_bits).reshape(tokens, H * D), mx.ROW, cu)
    np.testing.assert_array_equal(host(omx.data).reshape(tokens, H * D), q_ref)
    np.testing.assert_array_equal(host(omx.sf_compact), s_ref)
    comp, pad = unpack_packed(host(omx.sf_packed), mx.ROW, lens, H)
    np.testing.assert_array_equal(comp, s_ref)
    assert np.all(pad == 0x7F)
    oo, lo = oracle.method_fwd(f64(qb), f64(kb), f64(vb), cu, cu, scale, True, True, 128, THR)
    lse_h = host(lse)
    if not varlen:  # dense lse is [B][H][S]; the oracle's is [H][tokens]
        lse_h = lse_h.reshape(len(lens), H, lens[0]).transpose(1, 0, 2).reshape(H, tokens)
    check(f64(o_bits).reshape(tokens, H, D), lse_h, oo, lo)
