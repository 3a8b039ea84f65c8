"""GPU backward (tcgen05 kernel) vs the CPU oracle on the same seeded inputs.

Bar: dQ, dK, dV relative Frobenius <= 3e-2, for FP32 and FP16 (static scale)
dQ reduction.  Both sides receive the same O (bf16) and lse, produced by the
oracle's forward, so the backward is tested on its own; one case chains the
GPU forward into the GPU backward against the oracle's forward + backward.
"""
import math

import numpy as np
import pytest

import oracle
from mxfp8_block_scaled_fa_gb300 import inputs
from tests.helpers import f64, host, rel_fro, to_dev

pytestmark = pytest.mark.gpu

THR = 8.0
G_REL = 3e-2


@pytest.fixture(scope="module")
def mx():
    import torch
    from mxfp8_block_scaled_fa_gb300 import build, mxfa
    build.build()
    assert torch.cuda.is_available()
    return mxfa


def gpu_bwd(mx, qb, kb, vb, dob, o_bits, lse_dev, sq, sk, scale, causal, dq_mode=0, dq_static=1.0):
    import torch
    q = mx.quantize(to_dev(qb), mx.SQ, sq)
    k = mx.quantize(to_dev(kb), mx.SQ, sk)
    v = mx.quantize(to_dev(vb), mx.ROW, sk)
    do_t = to_dev(dob)
    dmx = mx.quantize(do_t, mx.SQ, sq)
    H, D = qb.shape[-2], qb.shape[-1]
    o_t = to_dev(o_bits).reshape(-1, H, D)
    dq, dk, dv = mx.attention_bwd(q, k, v, dmx, o_t, do_t.reshape(-1, H, D), lse_dev, sq, sk,
                                  scale, causal, dq_mode, dq_static)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    return [host(t.float()).astype(np.float64) for t in (dq, dk, dv)]


def oracle_fwd_out(qf, kf, vf, cu_q, cu_k, scale, causal):
    """The oracle forward's O and lse as the backward's interface carries them
    (O in bf16, lse in fp32): (O bits, O as float64, lse as float64).  Both
    backward implementations then receive exactly the same input values."""
    o, lse = oracle.method_fwd(qf, kf, vf, cu_q, cu_k, scale, causal, True, 128, THR)
    o_bits = inputs.f32_to_bf16_bits(o.astype(np.float32))
    return o_bits, inputs.bf16_bits_to_f32(o_bits).astype(np.float64), lse.astype(np.float32).astype(np.float64)


def check(got, ref, tag=""):
    errs = [rel_fro(g.reshape(r.shape), r) for g, r in zip(got, ref)]
    print(f"[bwd parity] {tag} rel-Fro dQ {errs[0]:.3e} dK {errs[1]:.3e} dV {errs[2]:.3e}")
    for name, e in zip(("dQ", "dK", "dV"), errs):
        assert e <= G_REL, f"{tag} {name} rel {e}"


@pytest.mark.parametrize("B,H,S,causal,dq_mode,dq_static", [
    (1, 2, 256, False, 0, 1.0),     # the tiny workload, fp32 dQ
    (1, 2, 256, False, 1, 1.0),     # fp16 dQ, static scale 1
    (1, 2, 256, False, 1, 16.0),    # fp16 dQ, static scale 2^4
    (1, 2, 384, True, 0, 1.0),
    (2, 2, 300, True, 0, 1.0),      # ragged tail in both key and query tiles
    (2, 3, 300, False, 1, 4.0),
    (1, 1, 33, False, 0, 1.0),
    (4, 20, 1000, True, 0, 1.0),    # more work items than SMs
])
def test_bwd_dense(mx, B, H, S, causal, dq_mode, dq_static):
    import torch
    D = 128
    scale = 1 / math.sqrt(D)
    qb, kb, vb, dob = inputs.dense_attn(B, H, S, D, seed=200 + S)
    f = lambda b: f64(b).reshape(B * S, H, D)
    cu = np.arange(0, (B + 1) * S, S, dtype=np.int32)
    o_bits, o_bf, lse = oracle_fwd_out(f(qb), f(kb), f(vb), cu, cu, scale, causal)
    lse_dense = lse.reshape(H, B, S).transpose(1, 0, 2).astype(np.float32)
    seqs = mx.Seqs.dense(B, S)
    got = gpu_bwd(mx, qb, kb, vb, dob, o_bits, torch.from_numpy(lse_dense.copy()).cuda(), seqs,
                  seqs, scale, causal, dq_mode, dq_static)
    ref = oracle.method_bwd(f(qb), f(kb), f(vb), f(dob), o_bf, lse, cu, cu, scale, causal, True)
    check(got, ref)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_varlen(mx, causal):
    import torch
    H, D = 2, 128
    lq = [64, 300, 7, 129, 1, 255]
    lk = lq if causal else [32, 200, 1, 260, 77, 128]
    qb, kb, vb, dob, cu_q, cu_k = inputs.varlen_attn(lq, lk, H, D, seed=31)
    scale = 1 / math.sqrt(D)
    o_bits, o_bf, lse = oracle_fwd_out(f64(qb), f64(kb), f64(vb), cu_q, cu_k, scale, causal)
    sq = mx.Seqs.varlen(lq, "cuda")
    sk = mx.Seqs.varlen(lk, "cuda")
    got = gpu_bwd(mx, qb, kb, vb, dob, o_bits, torch.from_numpy(lse.astype(np.float32)).cuda(),
                  sq, sk, scale, causal)
    ref = oracle.method_bwd(f64(qb), f64(kb), f64(vb), f64(dob), o_bf, lse, cu_q, cu_k, scale,
                            causal, True)
    check(got, ref)


def test_bwd_varlen_empty_sequences(mx):
    # keys of a sequence with no queries get dK = dV = 0; queries of a
    # sequence with no keys get dQ = 0 (their O is 0 and lse -inf)
    import torch
    H, D = 2, 128
    lq = [0, 70, 5, 130]
    lk = [40, 70, 0, 130]
    qb, kb, vb, dob, cu_q, cu_k = inputs.varlen_attn(lq, lk, H, D, seed=33)
    scale = 1 / math.sqrt(D)
    o_bits, o_bf, lse = oracle_fwd_out(f64(qb), f64(kb), f64(vb), cu_q, cu_k, scale, False)
    sq = mx.Seqs.varlen(lq, "cuda")
    sk = mx.Seqs.varlen(lk, "cuda")
    got = gpu_bwd(mx, qb, kb, vb, dob, o_bits, torch.from_numpy(lse.astype(np.float32)).cuda(),
                  sq, sk, scale, False)
    ref = oracle.method_bwd(f64(qb), f64(kb), f64(vb), f64(dob), o_bf, lse, cu_q, cu_k, scale,
                            False, True)
    for g, r in zip(got, ref):
        assert np.isfinite(g).all()
    no_key = np.repeat(np.asarray(lk) == 0, lq)
    no_query = np.repeat(np.asarray(lq) == 0, lk)
    assert np.all(got[0].reshape(-1, H, D)[no_key] == 0)
    assert np.all(got[1].reshape(-1, H, D)[no_query] == 0)
    assert np.all(got[2].reshape(-1, H, D)[no_query] == 0)
    check(got, ref)


def test_bwd_rows_outside_sequences(mx):
    # query tokens after the last sequence (total_q > cu_seqlens_q[nseq]) belong
    # to no sequence: their dQ rows are 0 whatever the workspace held before,
    # and the other rows are unchanged
    import dataclasses
    import torch
    H, D, extra = 2, 128, 24
    lq, lk = [70, 130], [90, 40]
    qb, kb, vb, dob, cu_q, cu_k = inputs.varlen_attn(lq, lk, H, D, seed=35)
    scale = 1 / math.sqrt(D)
    o_bits, o_bf, lse = oracle_fwd_out(f64(qb), f64(kb), f64(vb), cu_q, cu_k, scale, False)
    ref = oracle.method_bwd(f64(qb), f64(kb), f64(vb), f64(dob), o_bf, lse, cu_q, cu_k, scale,
                            False, True)
    total = sum(lq)
    sq = mx.Seqs.varlen(lq, "cuda")
    sk = mx.Seqs.varlen(lk, "cuda")
    sq_pad = dataclasses.replace(sq, total=total + extra)
    pad = lambda t: torch.cat([t, torch.zeros((extra,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)])
    q = mx.quantize(to_dev(qb), mx.SQ, sq)
    dmx = mx.quantize(to_dev(dob), mx.SQ, sq)
    q = mx.Mx(pad(q.data), q.sf_compact, q.sf_packed, q.blk)
    dmx = mx.Mx(pad(dmx.data), dmx.sf_compact, dmx.sf_packed, dmx.blk)
    k = mx.quantize(to_dev(kb), mx.SQ, sk)
    v = mx.quantize(to_dev(vb), mx.ROW, sk)
    o_t = pad(to_dev(o_bits).reshape(-1, H, D))
    do_t = pad(to_dev(dob).reshape(-1, H, D))
    lse_pad = np.concatenate([lse.reshape(H, total), np.zeros((H, extra))], axis=1).astype(np.float32)
    wsb = mx.mxfa_bwd_workspace_size(total + extra, sq.nseq, H, D, 0)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN bytes
    dq, dk, dv = mx.attention_bwd(q, k, v, dmx, o_t, do_t, torch.from_numpy(lse_pad).cuda(), sq_pad, sk,
                                  scale, False, ws=ws)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    got = [host(t.float()).astype(np.float64) for t in (dq, dk, dv)]
    assert np.all(got[0][total:] == 0)
    check([got[0][:total], got[1], got[2]], ref, "rows outside sequences")


@pytest.mark.parametrize("varlen", [False, True])
def test_bwd_constant_p_scale(mx, varlen):
    # P^T quantized with the constant scale 2^-8 instead of each block's own,
    # against the oracle in the same mode
    import torch
    H, D = 2, 128
    scale = 1 / math.sqrt(D)
    if varlen:
        lq = [64, 300, 7, 129, 1, 255]
        lk = [32, 200, 1, 260, 77, 128]
        qb, kb, vb, dob, cu_q, cu_k = inputs.varlen_attn(lq, lk, H, D, seed=71)
        sq, sk = mx.Seqs.varlen(lq, "cuda"), mx.Seqs.varlen(lk, "cuda")
        causal = False
    else:
        B, S = 2, 300
        qb, kb, vb, dob = (b.reshape(B * S, H, D) for b in inputs.dense_attn(B, H, S, D, seed=72))
        cu_q = cu_k = np.arange(0, (B + 1) * S, S, dtype=np.int32)
        sq = sk = mx.Seqs.dense(B, S)
        causal = True
    o_bits, o_bf, lse = oracle_fwd_out(f64(qb), f64(kb), f64(vb), cu_q, cu_k, scale, causal)
    lse_dev = (torch.from_numpy(lse.astype(np.float32)).cuda() if varlen else
               torch.from_numpy(lse.reshape(H, 2, 300).transpose(1, 0, 2).astype(np.float32)
                                .copy()).cuda())
    q = mx.quantize(to_dev(qb), mx.SQ, sq)
    k = mx.quantize(to_dev(kb), mx.SQ, sk)
    v = mx.quantize(to_dev(vb), mx.ROW, sk)
    do_t = to_dev(dob)
    dmx = mx.quantize(do_t, mx.SQ, sq)
    got = mx.attention_bwd(q, k, v, dmx, to_dev(o_bits), do_t, lse_dev, sq, sk, scale, causal,
                           opts=mx.AttnOpts(8.0, mx.P_SCALE_CONST))
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    ref = oracle.method_bwd(f64(qb), f64(kb), f64(vb), f64(dob), o_bf, lse, cu_q, cu_k, scale,
                            causal, True, 1)
    check([host(t.float()).astype(np.float64) for t in got], ref, "constant P scale")


def test_fwd_then_bwd_on_gpu(mx):
    # the path as a training step runs it: GPU forward output feeds the GPU backward
    import torch
    B, H, S, D = 1, 2, 256, 128
    scale = 1 / math.sqrt(D)
    qb, kb, vb, dob = inputs.dense_attn(B, H, S, D, seed=0)
    seqs = mx.Seqs.dense(B, S)
    q = mx.quantize(to_dev(qb), mx.ROW, seqs)
    k = mx.quantize(to_dev(kb), mx.ROW, seqs)
    v = mx.quantize(to_dev(vb), mx.COL, seqs)
    o, lse = mx.attention_fwd(q, k, v, seqs, seqs, scale, causal=True)
    do_t = to_dev(dob)
    dq, dk, dv = mx.attention_bwd(mx.quantize(to_dev(qb), mx.SQ, seqs),
                                  mx.quantize(to_dev(kb), mx.SQ, seqs),
                                  mx.quantize(to_dev(vb), mx.ROW, seqs),
                                  mx.quantize(do_t, mx.SQ, seqs), o, do_t.reshape(B * S, H, D),
                                  lse, seqs, seqs, scale, causal=True)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    f = lambda b: f64(b).reshape(B * S, H, D)
    # the forward against the oracle's forward, the backward against the
    # oracle's backward on the same O (bf16) and lse (fp32) that the GPU
    # backward received from the GPU forward
    from tests.test_gpu_fwd import check as fwd_check
    oo, lo = oracle.method_fwd(f(qb), f(kb), f(vb), None, None, scale, True, True, 128, THR)
    o_gpu = host(o.float()).astype(np.float64)
    lse_gpu = host(lse).reshape(H, B * S).astype(np.float64)
    fwd_check(o_gpu, lse_gpu, oo, lo)
    ref = oracle.method_bwd(f(qb), f(kb), f(vb), f(dob), o_gpu, lse_gpu, None, None, scale, True,
                            True)
    check([host(t.float()).astype(np.float64) for t in (dq, dk, dv)], ref, "chained")


@pytest.mark.parametrize("dq_mode,dq_static", [(0, 1.0), (1, 1.0)])
def test_bwd_llm_config_sampled_head(mx, dq_mode, dq_static):
    # the full LLM-shaped causal backward on the GPU, with FP32 and with FP16
    # (static scale) dQ accumulation; the oracle recomputes one (batch, head)
    # pair in full from the same O and lse
    import torch
    B, H, S, D = 2, 16, 8192, 128
    scale = 1 / math.sqrt(D)
    qb, kb, vb, dob = inputs.dense_attn(B, H, S, D, seed=1)
    b, h = 1, 5
    sl = lambda x: f64(x[b, :, h:h + 1, :])
    o_h_bits, o_h_bf, lse_h = oracle_fwd_out(sl(qb), sl(kb), sl(vb), None, None, scale, True)
    # O and lse for every head: the sampled head from the oracle, others from the GPU forward
    seqs = mx.Seqs.dense(B, S)
    q = mx.quantize(to_dev(qb), mx.ROW, seqs)
    k = mx.quantize(to_dev(kb), mx.ROW, seqs)
    v = mx.quantize(to_dev(vb), mx.COL, seqs)
    o, lse = mx.attention_fwd(q, k, v, seqs, seqs, scale, causal=True)
    torch.cuda.synchronize()
    o_bits = host(o.view(torch.int16)).view(np.uint16).reshape(B, S, H, D).copy()
    o_bits[b, :, h, :] = o_h_bits.reshape(S, D)
    lse_h32 = torch.from_numpy(lse_h.reshape(S).astype(np.float32)).cuda()  # already fp32 values
    lse.view(B, H, S)[b, h].copy_(lse_h32)
    got = gpu_bwd(mx, qb, kb, vb, dob, o_bits, lse, seqs, seqs, scale, True, dq_mode, dq_static)
    got = [g.reshape(B, S, H, D)[b, :, h:h + 1, :] for g in got]
    ref = oracle.method_bwd(sl(qb), sl(kb), sl(vb), sl(dob), o_h_bf, lse_h, None, None, scale, True,
                            True)
    check(got, ref, f"llm dq_mode {dq_mode}")


@pytest.mark.parametrize("varlen,dq_mode", [(False, 0), (False, 1), (True, 0)])
def test_bwd_mxfp8_gradients(mx, varlen, dq_mode):
    # the backward that also emits dQ, dK, dV as MXFP8 (1x32 blocks along D):
    # its bf16 dK and dV equal the plain backward's bit for bit (one CTA owns
    # each key row), and every MXFP8 payload and scale equals the oracle's ROW
    # quantization of the same call's bf16 gradient, byte for byte
    import torch
    from tests.helpers import unpack_packed
    H, D = 2, 128
    scale = 1 / math.sqrt(D)
    if varlen:
        lq = [64, 300, 7, 129, 1, 255]
        lk = [32, 200, 1, 260, 77, 128]
        qb, kb, vb, dob, cu_q, cu_k = inputs.varlen_attn(lq, lk, H, D, seed=51)
        sq, sk = mx.Seqs.varlen(lq, "cuda"), mx.Seqs.varlen(lk, "cuda")
        causal = False
    else:
        B, S = 2, 300
        lq = lk = [S] * B
        qb, kb, vb, dob = (b.reshape(B * S, H, D) for b in inputs.dense_attn(B, H, S, D, seed=52))
        cu_q = cu_k = np.arange(0, (B + 1) * S, S, dtype=np.int32)
        sq = sk = mx.Seqs.dense(B, S)
        causal = True
    o_bits, o_bf, lse = oracle_fwd_out(f64(qb), f64(kb), f64(vb), cu_q, cu_k, scale, causal)
    lse_dev = (torch.from_numpy(lse.astype(np.float32)).cuda() if varlen else
               torch.from_numpy(lse.reshape(H, len(lq), lq[0]).transpose(1, 0, 2).astype(np.float32)
                                .copy()).cuda())
    q = mx.quantize(to_dev(qb), mx.SQ, sq)
    k = mx.quantize(to_dev(kb), mx.SQ, sk)
    v = mx.quantize(to_dev(vb), mx.ROW, sk)
    do_t = to_dev(dob)
    dmx = mx.quantize(do_t, mx.SQ, sq)
    o_t = to_dev(o_bits)
    plain = mx.attention_bwd(q, k, v, dmx, o_t, do_t, lse_dev, sq, sk, scale, causal, dq_mode, 4.0)
    dq, dk, dv, dq_mx, dk_mx, dv_mx = mx.attention_bwd(q, k, v, dmx, o_t, do_t, lse_dev, sq, sk,
                                                       scale, causal, dq_mode, 4.0, grads_mx=True)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    bits = lambda t: host(t.view(torch.int16)).view(np.uint16)
    np.testing.assert_array_equal(bits(dk), bits(plain[1]))
    np.testing.assert_array_equal(bits(dv), bits(plain[2]))
    for name, g, m, lens, cu in (("dQ", dq, dq_mx, lq, cu_q), ("dK", dk, dk_mx, lk, cu_k),
                                 ("dV", dv, dv_mx, lk, cu_k)):
        gb = bits(g)
        tokens = gb.shape[0]
        q_ref, s_ref = oracle.quantize(f64(gb).reshape(tokens, H * D), mx.ROW, cu)
        np.testing.assert_array_equal(host(m.data).reshape(tokens, H * D), q_ref, err_msg=name)
        np.testing.assert_array_equal(host(m.sf_compact), s_ref, err_msg=name)
        comp, pad = unpack_packed(host(m.sf_packed), mx.ROW, lens, H)
        np.testing.assert_array_equal(comp, s_ref, err_msg=name)
        assert np.all(pad == 0x7F), name
    ref = oracle.method_bwd(f64(qb), f64(kb), f64(vb), f64(dob), o_bf, lse, cu_q, cu_k, scale, causal,
                            True)
    check([host(t.float()).astype(np.float64) for t in (dq, dk, dv)], ref, "mxfp8 grads")
