"""Pins for the oracle's attention forward and backward (CPU only).

Against: brute-force fp64 softmax attention, logsumexp, central finite
differences, invariants (constant V, causal row 0), a hand-worked row-sum
example (tests/golden/attn_rowsum.txt), inputs built so that the correct block
orientation is exact while any other orientation is not, and the equality of
packed (varlen) and per-sequence results.
"""
import math
import os

import numpy as np
import pytest

import oracle
from mxfp8_block_scaled_fa_gb300 import inputs

LOG2E = 1.0 / math.log(2.0)


def brute_fwd(q, k, v, scale, causal):
    """softmax(q k^T scale) v per head, fp64, one sequence [S, H, D]."""
    S, H, D = q.shape
    Sk = k.shape[0]
    o = np.zeros_like(q)
    lse = np.zeros((H, S))
    for h in range(H):
        s = q[:, h] @ k[:, h].T * scale
        if causal:
            s = np.where(np.arange(Sk)[None, :] > np.arange(S)[:, None], -np.inf, s)
        mx = s.max(axis=1, keepdims=True)
        e = np.exp(s - mx)
        o[:, h] = (e / e.sum(axis=1, keepdims=True)) @ v[:, h]
        lse[h] = (mx[:, 0] + np.log(e.sum(axis=1)))
    return o, lse


def _rand(shape, seed):
    return inputs.bf16_bits_to_f32(inputs.normal_bf16(shape, seed)).astype(np.float64)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,tile", [(37, 128), (300, 128), (300, 32)])
def test_fwd_quant_off_matches_brute_force(causal, S, tile):
    H, D = 2, 16
    q, k, v = (_rand((S, H, D), s) for s in (1, 2, 3))
    scale = 1 / math.sqrt(D)
    o, lse = oracle.attn_fwd(q, k, v, None, None, scale, causal, quant_p=False,
                             tile_n=tile)
    ob, lb = brute_fwd(q, k, v, scale, causal)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def test_fwd_lazy_rescale_is_exact_without_quantization():
    S, H, D = 300, 1, 32
    q, k, v = (_rand((S, H, D), s) for s in (4, 5, 6))
    q *= 3.0
    o0, l0 = oracle.attn_fwd(q, k, v, None, None, 0.2, False, False, 32, 0.0)
    o8, l8 = oracle.attn_fwd(q, k, v, None, None, 0.2, False, False, 32, 8.0)
    np.testing.assert_allclose(o8, o0, atol=1e-12)
    np.testing.assert_allclose(l8, l0, atol=1e-12)


def test_fwd_rowsum_golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "attn_rowsum.txt")
    vals = {}
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#") and "=" in line:
            key, expr = (t.strip() for t in line.split("=", 1))
            vals[key] = expr
    assert vals["o"] == "66/65" and vals["lse"] == "ln(65/32)"
    q = np.zeros((1, 1, 4)); q[0, 0, 0] = 1.0
    k = np.zeros((2, 1, 4)); k[1, 0, 0] = 2 * math.log(33 / 32)
    v = np.ones((2, 1, 4))
    cu_q = np.array([0, 1], np.int32); cu_k = np.array([0, 2], np.int32)
    o, lse = oracle.attn_fwd(q, k, v, cu_q, cu_k, 0.5, False, True)
    np.testing.assert_allclose(o, 66 / 65, rtol=1e-14)
    np.testing.assert_allclose(lse, math.log(65 / 32), rtol=1e-14)


def test_fwd_p_blocks_run_along_keys():
    # s' = -20 * ((j//32 + i) % 2): constant inside every 32-key block of a
    # row, alternating 1 / 2^-20 down a column.  Key-wise blocks are exact;
    # query-wise blocks would flush the 2^-20 entries (2^-12 < 2^-10).
    S, H, D = 128, 1, 2
    scale = 1.0
    c = -20.0 / (scale * LOG2E)
    j = np.arange(S)
    q = np.zeros((S, H, D)); q[0::2, 0, 0] = 1.0; q[1::2, 0, 1] = 1.0
    k = np.zeros((S, H, D))
    k[:, 0, 0] = np.where((j // 32) % 2 == 0, 0.0, c)
    k[:, 0, 1] = np.where((j // 32) % 2 == 1, 0.0, c)
    v = _rand((S, H, D), 9)
    oq, lq = oracle.attn_fwd(q, k, v, None, None, scale, False, True)
    o0, l0 = oracle.attn_fwd(q, k, v, None, None, scale, False, False)
    np.testing.assert_allclose(oq, o0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lq, l0, rtol=0, atol=1e-13)


def test_fwd_invariants_with_quantization():
    S, H, D = 256, 2, 128
    q, k = _rand((S, H, D), 10), _rand((S, H, D), 11)
    v = np.ones((S, H, D))
    scale = 1 / math.sqrt(D)
    for causal in (False, True):
        o, _ = oracle.attn_fwd(q, k, v, None, None, scale, causal, True)
        # rows of softmax sum to 1 up to the E4M3 rounding of P (half a
        # quantum: at most 2^-4 relative for normal values, tiny ones below)
        assert np.max(np.abs(o - 1.0)) < 2.0 ** -4
        assert np.max(np.abs(o - 1.0)) > 0  # P really is quantized
    vq = oracle.qdq(_rand((S, H, D), 12), oracle.COL)
    o, _ = oracle.attn_fwd(q, k, vq, None, None, scale, True, True)
    np.testing.assert_array_equal(o[0], vq[0])  # causal row 0 returns V^_0


def test_fwd_varlen_equals_per_sequence():
    H, D = 2, 32
    lq, lk = [5, 130, 64], [40, 7, 129]
    q, k, v, _, cu_q, cu_k = inputs.varlen_attn(lq, lk, H, D, 13)
    f = lambda b: inputs.bf16_bits_to_f32(b).astype(np.float64)
    q, k, v = f(q), f(k), f(v)
    o, lse = oracle.method_fwd(q, k, v, cu_q, cu_k, 0.125, False, True)
    for g in range(3):
        sq = slice(cu_q[g], cu_q[g + 1]); sk = slice(cu_k[g], cu_k[g + 1])
        og, lg = oracle.method_fwd(q[sq], k[sk], v[sk], None, None, 0.125, False, True)
        np.testing.assert_array_equal(o[sq], og)
        np.testing.assert_array_equal(lse[:, sq], lg)


def test_empty_key_sequence_gives_zero_output_and_neg_inf_lse():
    # a query whose key sequence is empty attends to nothing: O = 0, lse = -inf
    # (the empty softmax sum); the other sequences are unaffected, and the
    # backward gives dQ = 0 for such queries and dK = dV = 0 for keys of a
    # sequence without queries
    H, D = 2, 32
    lq, lk = [3, 0, 40], [0, 9, 33]
    q, k, v, do, cu_q, cu_k = inputs.varlen_attn(lq, lk, H, D, 17)
    f = lambda b: inputs.bf16_bits_to_f32(b).astype(np.float64)
    q, k, v, do = f(q), f(k), f(v), f(do)
    o, lse = oracle.method_fwd(q, k, v, cu_q, cu_k, 0.2, False, True)
    assert np.all(o[:3] == 0.0) and np.all(np.isneginf(lse[:, :3]))
    og, lg = oracle.method_fwd(q[3:], k[9:], v[9:], None, None, 0.2, False, True)
    np.testing.assert_array_equal(o[3:], og)
    np.testing.assert_array_equal(lse[:, 3:], lg)
    dq, dk, dv = oracle.method_bwd(q, k, v, do, o, lse, cu_q, cu_k, 0.2, False, True)
    assert np.all(dq[:3] == 0.0)
    assert np.all(dk[:9] == 0.0) and np.all(dv[:9] == 0.0)
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()


# ---------------------------------------------------------------- backward
def _loss_grads_fd(q, k, v, do, scale, causal, h=1e-6):
    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd(q_, k_, v_, None, None, scale, causal, False)
        return float(np.sum(o * do))
    grads = []
    for which in range(3):
        base = [q, k, v]
        g = np.zeros_like(base[which])
        it = np.nditer(g, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in base]; minus = [a.copy() for a in base]
            plus[which][idx] += h; minus[which][idx] -= h
            g[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        grads.append(g)
    return grads


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_quant_off_matches_finite_differences(causal):
    S, H, D = 12, 1, 8
    q, k, v, do = (_rand((S, H, D), s) for s in (20, 21, 22, 23))
    scale = 1 / math.sqrt(D)
    o, lse = oracle.attn_fwd(q, k, v, None, None, scale, causal, False)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, o, do, lse, None, None, scale, causal,
                                 False, False)
    fq, fk, fv = _loss_grads_fd(q, k, v, do, scale, causal)
    for a, b in ((dq, fq), (dk, fk), (dv, fv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=2e-8)


def test_bwd_p_blocks_run_along_queries():
    # P_ij = 2^(-20 (j % 2)) (constant along queries, alternating along keys):
    # query-wise 1x32 blocks are exact; key-wise blocks would zero odd keys.
    S, H, D = 64, 1, 4
    scale = 0.5
    c = -20.0 * math.log(2.0) / scale
    q = np.zeros((S, H, D)); q[:, 0, 0] = 1.0
    k = np.zeros((S, H, D)); k[1::2, 0, 0] = c
    v = _rand((S, H, D), 30); do = _rand((S, H, D), 31)
    lse = np.zeros((H, S)); zeros = np.zeros((S, H, D))
    _, _, dvq = oracle.attn_bwd(q, k, v, do, zeros, do, lse, None, None, scale,
                                False, True, False)
    _, _, dv0 = oracle.attn_bwd(q, k, v, do, zeros, do, lse, None, None, scale,
                                False, False, False)
    np.testing.assert_allclose(dvq, dv0, rtol=1e-13, atol=0)
    expect_odd = 2.0 ** -20 * do.sum(axis=0)
    np.testing.assert_allclose(dvq[1], expect_odd, rtol=1e-13)


@pytest.mark.parametrize("vary", ["queries", "keys"])
def test_bwd_ds_blocks_are_square(vary):
    # P = 1 (S = 0, lse = 0), Delta = 0 (O = 0), dS_ij = dP_ij = a_i or b_j with
    # values alternating 1 / 2^-20.  A 32x32 block holding both flushes the
    # 2^-20 entries (2^-12 < 2^-10); row-only or column-only blocks would not.
    L, H, D = 64, 1, 4
    scale = 0.25
    t = np.where(np.arange(L) % 2 == 0, 1.0, 2.0 ** -20)
    q = np.zeros((L, H, D)); q[:, 0, 0] = 1.0
    k = np.zeros((L, H, D)); k[:, 0, 1] = 1.0
    v = np.zeros((L, H, D)); do = np.zeros((L, H, D))
    if vary == "queries":
        do[:, 0, 0] = t; v[:, 0, 0] = 1.0
    else:
        do[:, 0, 0] = 1.0; v[:, 0, 0] = t
    lse = np.zeros((H, L)); zeros = np.zeros((L, H, D))
    dq, dk, _ = oracle.attn_bwd(q, k, v, do, zeros, do, lse, None, None, scale,
                                False, True, True)
    even = (np.arange(L) % 2 == 0).astype(float)
    if vary == "queries":  # dS^_ij = 1 for even i else 0
        exp_dk0 = scale * even.sum() * np.ones(L)
        exp_dq1 = scale * L * even
    else:                  # dS^_ij = 1 for even j else 0
        exp_dk0 = scale * L * even
        exp_dq1 = scale * even.sum() * np.ones(L)
    np.testing.assert_allclose(dk[:, 0, 0], exp_dk0, rtol=1e-14, atol=0)
    np.testing.assert_allclose(dq[:, 0, 1], exp_dq1, rtol=1e-14, atol=0)
    assert np.all(dk[:, 0, 1:] == 0) and np.all(dq[:, 0, [0, 2, 3]] == 0)


def test_bwd_varlen_equals_per_sequence():
    H, D = 2, 32
    lens = [45, 100, 33]
    q, k, v, do, cu, _ = inputs.varlen_attn(lens, lens, H, D, 40)
    f = lambda b: inputs.bf16_bits_to_f32(b).astype(np.float64)
    q, k, v, do = f(q), f(k), f(v), f(do)
    o, lse = oracle.method_fwd(q, k, v, cu, cu, 0.2, True, True)
    got = oracle.method_bwd(q, k, v, do, o, lse, cu, cu, 0.2, True, True)
    for g in range(3):
        s = slice(cu[g], cu[g + 1])
        og, lg = oracle.method_fwd(q[s], k[s], v[s], None, None, 0.2, True, True)
        ref = oracle.method_bwd(q[s], k[s], v[s], do[s], og, lg, None, None, 0.2,
                                True, True)
        for a, b in zip(got, ref):
            np.testing.assert_array_equal(a[s], b)


def test_bwd_quantized_close_to_exact():
    # sanity of magnitude: the quantized method stays near exact attention
    S, H, D = 256, 1, 128
    q, k, v, do = (_rand((S, H, D), s) for s in (50, 51, 52, 53))
    scale = 1 / math.sqrt(D)
    o, lse = oracle.method_fwd(q, k, v, None, None, scale, True, False)
    ex = oracle.method_bwd(q, k, v, do, o, lse, None, None, scale, True, False)
    qu = oracle.method_bwd(q, k, v, do, o, lse, None, None, scale, True, True)
    for a, b in zip(qu, ex):
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        assert 1e-3 < rel < 0.15


# ----------------------------------------------------- constant P scale mode
def _one_hot_fwd(p_scale, lazy_thr):
    # one query (q = 1), 64 keys with scores s'_j = k_j (scale ln 2 makes
    # scale * log2 e = 1 exactly), V_j = e_j so that O_j = P^_j / l
    keys = np.full(64, -40.0)
    keys[0] = 0.0                        # block 0: P~ = 1 (the row maximum)
    keys[1:32] = -30.0
    keys[32], keys[33], keys[34] = -10.0, -18.0, -11.0   # block 1: max 2^-10
    v = np.eye(64).reshape(64, 1, 64)
    qq = np.zeros((1, 1, 64)); qq[0, 0, 0] = 1.0
    kk = np.zeros((64, 1, 64)); kk[:, 0, 0] = keys
    o, lse = oracle.attn_fwd(qq, kk, v, np.array([0, 1], np.int32), np.array([0, 64], np.int32),
                             math.log(2.0), False, True, 128, lazy_thr, p_scale)
    l = 1 + 31 * 2.0 ** -30 + 2.0 ** -10 + 2.0 ** -18 + 2.0 ** -11 + 29 * 2.0 ** -40
    return o[0, 0] * l


def test_constant_p_scale_forward_worked_example():
    # dynamic block scales: block 1 (max 2^-10) takes 2^-18, so 2^-18 is kept
    # exactly; the constant scale (exact rescale, threshold 0 -> 2^-8) puts
    # 2^-18 at 2^-10 on the E4M3 grid, half the smallest subnormal 2^-9: a tie
    # that rounds to the even code 0.  2^-10 -> 0.25 and 2^-11 -> 0.125 stay exact.
    pd = _one_hot_fwd(0, 0.0)
    pc = _one_hot_fwd(1, 0.0)
    for p in (pd, pc):
        assert abs(p[0] - 1.0) < 1e-15
        assert abs(p[32] - 2.0 ** -10) < 1e-18 and abs(p[34] - 2.0 ** -11) < 1e-18
        assert np.all(np.abs(p[1:32]) < 1e-20)   # 2^-30 flushes in both modes
    assert abs(pd[33] - 2.0 ** -18) < 1e-20
    assert pc[33] == 0.0
    # the lazy threshold 8 makes the constant exponent 0 (the largest possible
    # P~ = 2^8 -> 256): 2^-10 is then half the smallest E4M3 step 2^-9, a tie
    # to the even code 0, and 2^-11, 2^-18 lie below it -- block 1 vanishes
    p8 = _one_hot_fwd(1, 8.0)
    assert abs(p8[0] - 1.0) < 1e-15
    assert p8[32] == 0.0 and p8[33] == 0.0 and p8[34] == 0.0


def test_constant_p_scale_backward_worked_example():
    # one key (S = 0), 32 queries with lse_i chosen so that P_i = exp(-lse_i):
    # P = (2^-10, 2^-19, rest 2^-10); dO_i = e_i so that dV[i] = P^_i.  The
    # dynamic block scale 2^-18 keeps 2^-19 (0.5 on the E4M3 grid); the
    # constant scale 2^-8 puts it at 2^-11, below half of 2^-9: zero
    L = 32
    q = np.zeros((L, 1, 1)); k = np.zeros((1, 1, 1))
    v = np.zeros((1, 1, L)); do = np.eye(L).reshape(L, 1, L)
    o = np.zeros((L, 1, L))
    p = np.full(L, 2.0 ** -10); p[1] = 2.0 ** -19
    lse = (-np.log(p)).reshape(1, L)
    cq, ck = np.array([0, L], np.int32), np.array([0, 1], np.int32)
    qd = np.zeros((L, 1, L)); kd = np.zeros((1, 1, L))
    _, _, dv_d = oracle.attn_bwd(qd, kd, v, do, o, do, lse, cq, ck, 1.0, False, True, False, 0)
    _, _, dv_c = oracle.attn_bwd(qd, kd, v, do, o, do, lse, cq, ck, 1.0, False, True, False, 1)
    np.testing.assert_allclose(dv_d[0, 0, 1], 2.0 ** -19, rtol=1e-12)
    assert dv_c[0, 0, 1] == 0.0
    np.testing.assert_allclose(dv_c[0, 0, [0, 2, 31]], 2.0 ** -10, rtol=1e-12)
    np.testing.assert_allclose(dv_d[0, 0, [0, 2, 31]], 2.0 ** -10, rtol=1e-12)


def test_delta_from_the_quantized_do():
    # With a single key the softmax is the constant 1, so the exact gradients
    # with respect to Q and K vanish.  The method keeps that exactly when
    # Delta takes the same dequantized dO^ as dP: with V and O exact (small
    # integers survive every block scale), dP = dO^ . V = dO^ . O = Delta and
    # dS = 0.  Taking Delta from the bf16 dO instead (1 + 2^-6 rounds to 1 in
    # E4M3) leaves dS = P (dO^ - dO) . V != 0.
    D = 32
    q = np.zeros((1, 1, D)); q[0, 0, :4] = [1.0, -2.0, 3.0, 1.0]
    k = np.zeros((1, 1, D)); k[0, 0, :4] = [2.0, 1.0, -1.0, 4.0]
    v = np.zeros((1, 1, D)); v[0, 0, :4] = [3.0, -1.0, 2.0, 1.0]
    do = np.zeros((1, 1, D)); do[0, 0, :4] = 1.0 + 2.0 ** -6
    o, lse = oracle.method_fwd(q, k, v, None, None, 0.25, False, True)
    np.testing.assert_array_equal(o, v)   # one key: O = V exactly
    dq, dk, dv = oracle.method_bwd(q, k, v, do, o, lse, None, None, 0.25, False, True)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    dos = oracle.qdq(do, 2)
    assert dos[0, 0, 0] == 1.0
    dq0, dk0, _ = oracle.attn_bwd(oracle.qdq(q, 2), oracle.qdq(k, 2), oracle.qdq(v, 0), dos, o, do, lse,
                                  None, None, 0.25, False, True, True)
    assert np.abs(dq0).max() > 0 and np.abs(dk0).max() > 0


def test_backward_p_clamped_at_one():
    # One query, three keys, D = 1, scale 1: S = (2, 0.5, -1) with lse = 1
    # given (smaller than the first score, as a recompute from other operands
    # can make it).  Exact attention never has P > 1, so the first key takes
    # P = 1 (not e), the others exp(S - lse).  With dO = 1, O = 0 and no
    # quantization, dV_j = P_j.
    q = np.ones((1, 1, 1))
    k = np.array([2.0, 0.5, -1.0]).reshape(3, 1, 1)
    v = np.zeros((3, 1, 1))
    do = np.ones((1, 1, 1))
    o = np.zeros((1, 1, 1))
    lse = np.ones((1, 1))
    _, _, dv = oracle.attn_bwd(q, k, v, do, o, do, lse, None, None, 1.0, False, False, False)
    assert dv[0, 0, 0] == 1.0
    assert abs(dv[1, 0, 0] - math.exp(-0.5)) <= 1e-15
    assert abs(dv[2, 0, 0] - math.exp(-2.0)) <= 1e-15


def test_results_do_not_depend_on_thread_count():
    # every output element keeps its own summation order, so the oracle's
    # results are bit-identical on one host thread and on all of them
    q, k, v, do = (_rand((96, 2, 128), s) for s in (70, 71, 72, 73))
    scale = 1 / math.sqrt(128)
    cores = oracle.num_threads()
    runs = []
    for n in (1, cores):
        oracle.set_num_threads(n)
        o, lse = oracle.method_fwd(q, k, v, None, None, scale, True, True, 128, 8.0)
        g = oracle.method_bwd(q, k, v, do, o, lse, None, None, scale, True, True)
        runs.append((o, lse) + tuple(g))
    oracle.set_num_threads(cores)
    for a, b in zip(*runs):
        np.testing.assert_array_equal(a, b)
