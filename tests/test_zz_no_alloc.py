"""mxfa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (allocator hooks, runtimes that forbid cudaMalloc after start-up,
bindings without a device allocator).  Instead of a caller workspace it uses
a scratch array built into the library.  Checked through the C ABI against
mxfa_bwd with a caller-provided workspace, on two calls in a row: dK and dV
bit for bit (one CTA owns each key row, in a fixed order), dQ to within the
reduction order of its accumulator (1e-5 relative with fp32 accumulation, a
few fp16 spacings with fp16), and all three against the oracle at the
backward pass's bar (relative Frobenius <= 3e-2).

Collected last on purpose: a run that stops at the first failure has run
every other test before this one.
"""
import ctypes
import math

import numpy as np
import pytest

import oracle
from mxfp8_block_scaled_fa_gb300 import inputs
from tests.helpers import f64, host, rel_fro, to_dev

pytestmark = pytest.mark.gpu

G_REL = 3e-2


@pytest.fixture(scope="module")
def mx():
    import torch
    from mxfp8_block_scaled_fa_gb300 import build, mxfa
    build.build()
    assert torch.cuda.is_available()
    return mxfa


def _prepare(mx, seed, causal, S):
    B, H, D = 1, 2, 128
    scale = 1 / math.sqrt(D)
    qb, kb, vb, dob = inputs.dense_attn(B, H, S, D, seed=seed)
    seqs = mx.Seqs.dense(B, S)
    q, k, v = (to_dev(x) for x in (qb, kb, vb))
    do = to_dev(dob).reshape(B * S, H, D)
    o, lse = mx.attention_fwd(mx.quantize(q, mx.ROW, seqs), mx.quantize(k, mx.ROW, seqs),
                              mx.quantize(v, mx.COL, seqs), seqs, seqs, scale, causal)
    ops = (mx.quantize(q, mx.SQ, seqs), mx.quantize(k, mx.SQ, seqs), mx.quantize(v, mx.ROW, seqs),
           mx.quantize(do, mx.SQ, seqs))
    return dict(B=B, H=H, S=S, D=D, scale=scale, seqs=seqs, ops=ops, o=o, lse=lse, do=do,
                bits=(qb, kb, vb, dob))


def test_noalloc_matches_workspace_backward_twice(mx):
    import torch
    assert mx.lib().mxfa_bwd_noalloc_scratch_bytes() == 32 << 20
    # two calls in a row: different inputs, sizes, masking and dQ precision, so
    # the second call also shows that nothing left in the shared scratch leaks in
    for seed, causal, dq_mode, dq_static, S in ((0, False, 0, 1.0, 384), (7, True, 1, 16.0, 256)):
        c = _prepare(mx, seed, causal, S)
        q, k, v, dmx = c["ops"]
        ref = mx.attention_bwd(q, k, v, dmx, c["o"], c["do"], c["lse"], c["seqs"], c["seqs"],
                               c["scale"], causal, dq_mode, dq_static)
        got = [torch.empty_like(t) for t in ref]
        mx.mxfa_bwd_noalloc(q.mx_in(), k.mx_in(), v.mx_in(), dmx.mx_in(), c["o"], c["do"],
                            c["lse"], c["B"], c["S"], c["H"], c["D"], c["scale"], causal,
                            dq_mode, dq_static, got[0], got[1], got[2])
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        bits = lambda t: host(t.view(torch.int16))
        for name, g, r in zip(("dK", "dV"), got[1:], ref[1:]):
            np.testing.assert_array_equal(bits(g), bits(r), err_msg=name)
        gq, rq = host(got[0].float()).astype(np.float64), host(ref[0].float()).astype(np.float64)
        assert np.isfinite(gq).all()
        # the accumulators may sum the key tiles' partials in another order;
        # the bf16 dQ then differs by at most one bf16 rounding step (fp32
        # accumulation, sums equal to ~1e-7) or two plus a few fp16 spacings
        # of the static-scaled accumulator (fp16 accumulation)
        e = np.floor(np.log2(np.maximum(np.abs(rq), 2.0 ** -126)))
        tol = 2.0 ** (e - 7) if dq_mode == 0 else 2.0 ** (e - 6) + 4 * 2.0 ** -24 / dq_static
        assert np.all(np.abs(gq - rq) <= tol), np.max(np.abs(gq - rq) - tol)
        assert rel_fro(gq, rq) <= (1e-4 if dq_mode == 0 else 1e-2), rel_fro(gq, rq)
        # and against the oracle's backward on the same O and lse
        B, H, S, D = c["B"], c["H"], c["S"], c["D"]
        qb, kb, vb, dob = c["bits"]
        f = lambda x: f64(x).reshape(B * S, H, D)
        o_bf = host(c["o"].float()).astype(np.float64).reshape(B * S, H, D)
        lse_o = host(c["lse"]).reshape(H, B * S).astype(np.float64)
        want = oracle.method_bwd(f(qb), f(kb), f(vb), f(dob), o_bf, lse_o, None, None, c["scale"],
                                 causal, True)
        for name, g, w in zip(("dQ", "dK", "dV"), got, want):
            gg = host(g.float()).astype(np.float64).reshape(w.shape)
            assert rel_fro(gg, w) <= G_REL, (name, rel_fro(gg, w))


def test_noalloc_checks_arguments_before_its_scratch_size(mx):
    # a bad call gets the same status as from mxfa_bwd, even when the problem
    # would also be too large for the scratch array
    m = mx.MxIn(0x1000, 0x2000)
    r = ctypes.byref
    args = lambda D, o: (r(m), r(m), r(m), r(m), o, 0x5000, 0x6000, 2, 8192, 16, D, 0.088, 1, 0,
                         1.0, 0x7000, 0x8000, 0x9000, None)
    assert mx.lib().mxfa_bwd_noalloc(*args(64, 0x4000)) == 2     # MXFA_ERR_UNSUPPORTED (D)
    assert mx.lib().mxfa_bwd_noalloc(*args(128, None)) == 1      # MXFA_ERR_INVALID_ARG (o)
    assert mx.lib().mxfa_bwd_noalloc(*args(128, 0x4008)) == 3    # MXFA_ERR_MISALIGNED (o)


def test_noalloc_rejects_problems_beyond_its_scratch(mx):
    # B2 S8192 H16 needs ~129 MiB of workspace: refused before any pointer is used
    m = mx.MxIn(0x1000, 0x2000)
    r = ctypes.byref
    st = mx.lib().mxfa_bwd_noalloc(r(m), r(m), r(m), r(m), 0x4000, 0x5000, 0x6000, 2, 8192, 16,
                                   128, 0.088, 1, 0, 1.0, 0x7000, 0x8000, 0x9000, None)
    assert st == 4  # MXFA_ERR_WORKSPACE_TOO_SMALL
