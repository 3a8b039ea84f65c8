"""mxfa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (allocator hooks, runtimes that forbid cudaMalloc after start-up,
bindings without a device allocator).  Instead of a caller workspace it uses
a scratch array built into the library.  Checked through the C ABI against
mxfa_bwd with a caller-provided workspace, on two calls in a row, at the
backward pass's tolerance (relative Frobenius <= 3e-2).

Collected last on purpose: a run that stops at the first failure has run
every other test before this one.
"""
import ctypes
import math

import numpy as np
import pytest

from mxfp8_block_scaled_fa_gb300 import inputs
from tests.helpers import host, rel_fro, to_dev

pytestmark = pytest.mark.gpu

G_REL = 3e-2


@pytest.fixture(scope="module")
def mx():
    import torch
    from mxfp8_block_scaled_fa_gb300 import build, mxfa
    build.build()
    assert torch.cuda.is_available()
    return mxfa


def _prepare(mx, seed, causal):
    B, H, S, D = 1, 2, 256, 128
    scale = 1 / math.sqrt(D)
    qb, kb, vb, dob = inputs.dense_attn(B, H, S, D, seed=seed)
    seqs = mx.Seqs.dense(B, S)
    q, k, v = (to_dev(x) for x in (qb, kb, vb))
    do = to_dev(dob).reshape(B * S, H, D)
    o, lse = mx.attention_fwd(mx.quantize(q, mx.ROW, seqs), mx.quantize(k, mx.ROW, seqs),
                              mx.quantize(v, mx.COL, seqs), seqs, seqs, scale, causal)
    ops = (mx.quantize(q, mx.SQ, seqs), mx.quantize(k, mx.SQ, seqs), mx.quantize(v, mx.ROW, seqs),
           mx.quantize(do, mx.SQ, seqs))
    return dict(B=B, H=H, S=S, D=D, scale=scale, seqs=seqs, ops=ops, o=o, lse=lse, do=do)


def test_noalloc_matches_workspace_backward_twice(mx):
    import torch
    assert mx.lib().mxfa_bwd_noalloc_scratch_bytes() == 32 << 20
    # two calls in a row: different inputs, masking and dQ precision, so the
    # second call also shows that nothing left in the shared scratch leaks in
    for seed, causal, dq_mode, dq_static in ((0, False, 0, 1.0), (7, True, 1, 16.0)):
        c = _prepare(mx, seed, causal)
        q, k, v, dmx = c["ops"]
        ref = mx.attention_bwd(q, k, v, dmx, c["o"], c["do"], c["lse"], c["seqs"], c["seqs"],
                               c["scale"], causal, dq_mode, dq_static)
        got = [torch.empty_like(t) for t in ref]
        mx.mxfa_bwd_noalloc(q.mx_in(), k.mx_in(), v.mx_in(), dmx.mx_in(), c["o"], c["do"],
                            c["lse"], c["B"], c["S"], c["H"], c["D"], c["scale"], causal,
                            dq_mode, dq_static, got[0], got[1], got[2])
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            gg, rr = host(g.float()), host(r.float())
            assert np.isfinite(gg).all(), name
            assert rel_fro(gg, rr) <= G_REL, (name, rel_fro(gg, rr))


def test_noalloc_rejects_problems_beyond_its_scratch(mx):
    # B2 S8192 H16 needs ~129 MiB of workspace: refused before any pointer is used
    m = mx.MxIn(0x1000, 0x2000)
    r = ctypes.byref
    st = mx.lib().mxfa_bwd_noalloc(r(m), r(m), r(m), r(m), 0x4000, 0x5000, 0x6000, 2, 8192, 16,
                                   128, 0.088, 1, 0, 1.0, 0x7000, 0x8000, 0x9000, None)
    assert st == 4  # MXFA_ERR_WORKSPACE_TOO_SMALL
