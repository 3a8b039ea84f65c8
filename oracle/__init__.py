"""CPU oracle for MXFP8 block-scaled attention -- TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 C (``mxfa_oracle.c``) behind ctypes.  Only the tests, the
smoke check and the benchmark's CPU-baseline / reference leg may import this
package; the product path never does and shares no code with it.

Layouts: attention tensors are token-major ``[tokens, H, D]`` float64 (dense
``[B, S, H, D]`` is the varlen layout with uniform ``cu_seqlens``); the
log-sum-exp is ``[H, tokens]``.  Quantized tensors are treated as 2-D
``[tokens, H*D]`` so that 1x32 row blocks and 32x32 square blocks stay inside
one head and 32x1 column blocks run along the tokens of one sequence.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

ROW, COL, SQ = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmxfa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, OpenMP, no FP contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64, I32, D = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.mxo_e4m3_decode.restype = D
            lib.mxo_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.mxo_e4m3_encode.restype = ctypes.c_uint8
            lib.mxo_e4m3_encode.argtypes = [D]
            lib.mxo_e8m0_from_amax.restype = ctypes.c_uint8
            lib.mxo_e8m0_from_amax.argtypes = [D]
            lib.mxo_e8m0_decode.restype = D
            lib.mxo_e8m0_decode.argtypes = [ctypes.c_uint8]
            lib.mxo_quantize.restype = None
            lib.mxo_quantize.argtypes = [P, I64, I64, I32, P, I32, P, P]
            lib.mxo_dequantize.restype = None
            lib.mxo_dequantize.argtypes = [P, P, I64, I64, I32, P, I32, P]
            lib.mxo_attn_fwd.restype = None
            lib.mxo_attn_fwd.argtypes = [P, P, P, P, P, I32, I32, I32, D, I32, I32,
                                         I32, D, P, P, I64, I32]
            lib.mxo_attn_bwd.restype = None
            lib.mxo_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I32, I32, I32, D,
                                         I32, I32, I32, P, P, P, I64, I32]
            lib.mxo_rmsnorm_quant.restype = None
            lib.mxo_rmsnorm_quant.argtypes = [P, P, I64, I64, ctypes.c_float, I32,
                                              ctypes.c_int32, P, P, P, P, P, P, P]
            lib.mxo_fp_decode.restype = D
            lib.mxo_fp_decode.argtypes = [I32, ctypes.c_uint8]
            lib.mxo_fp_encode.restype = ctypes.c_uint8
            lib.mxo_fp_encode.argtypes = [I32, D]
            lib.mxo_fp_max.restype = D
            lib.mxo_fp_max.argtypes = [I32]
            lib.mxo_quantize_mx.restype = None
            lib.mxo_quantize_mx.argtypes = [P, I64, I64, I32, P, P]
            lib.mxo_quantize_nvfp4.restype = D
            lib.mxo_quantize_nvfp4.argtypes = [P, I64, I64, P, P]
            lib.mxo_gemm_nt.restype = None
            lib.mxo_gemm_nt.argtypes = [P, P, I64, I64, I64, P]
            lib.mxo_num_threads.restype = I32
            lib.mxo_num_threads.argtypes = []
            lib.mxo_set_num_threads.restype = None
            lib.mxo_set_num_threads.argtypes = [I32]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().mxo_num_threads())


def set_num_threads(n: int) -> None:
    """Host threads for later calls (results do not depend on the count)."""
    _load().mxo_set_num_threads(int(n))


# ---------------------------------------------------------------- codecs
def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.mxo_e4m3_decode(int(v)) for v in c.ravel()]).reshape(c.shape)


def e4m3_encode(vals) -> np.ndarray:
    lib = _load()
    v = np.asarray(vals, dtype=np.float64)
    return np.array([lib.mxo_e4m3_encode(float(x)) for x in v.ravel()],
                    dtype=np.uint8).reshape(v.shape)


def e8m0_from_amax(amax: float) -> int:
    return int(_load().mxo_e8m0_from_amax(float(amax)))


def e8m0_decode(s: int) -> float:
    return float(_load().mxo_e8m0_decode(int(s)))


# ------------------------------------------------------------- quantizer
def _seg(rows, cu):
    if cu is None:
        cu = np.array([0, rows], dtype=np.int32)
    cu = _c(cu, np.int32)
    return cu, len(cu) - 1


def sf_rows(cu, rows) -> int:
    """Number of compact 32-row scale rows for column/square blocks."""
    cu, n = _seg(rows, cu)
    return int(sum((int(cu[i + 1]) - int(cu[i]) + 31) // 32 for i in range(n)))


def quantize(x2d, mode: int, cu=None):
    """Quantize x[rows, cols] (float64) -> (payload u8[rows, cols], compact SF)."""
    lib = _load()
    x = _c(x2d, np.float64)
    rows, cols = x.shape
    cu_, n = _seg(rows, cu)
    q = np.zeros((rows, cols), np.uint8)
    if mode == ROW:
        sf = np.zeros((rows, cols // 32), np.uint8)
    elif mode == COL:
        sf = np.zeros((sf_rows(cu_, rows), cols), np.uint8)
    else:
        sf = np.zeros((sf_rows(cu_, rows), cols // 32), np.uint8)
    lib.mxo_quantize(_ptr(x), rows, cols, mode, _ptr(cu_), n, _ptr(q), _ptr(sf))
    return q, sf


def dequantize(q, sf, mode: int, cu=None) -> np.ndarray:
    lib = _load()
    q = _c(q, np.uint8)
    sf = _c(sf, np.uint8)
    rows, cols = q.shape
    cu_, n = _seg(rows, cu)
    x = np.zeros((rows, cols), np.float64)
    lib.mxo_dequantize(_ptr(q), _ptr(sf), rows, cols, mode, _ptr(cu_), n, _ptr(x))
    return x


def qdq(x3d, mode: int, cu=None) -> np.ndarray:
    """Quantize then dequantize a [tokens, H, D] tensor (as [tokens, H*D])."""
    t, h, d = x3d.shape
    q, sf = quantize(np.asarray(x3d, np.float64).reshape(t, h * d), mode, cu)
    return dequantize(q, sf, mode, cu).reshape(t, h, d)


# ------------------------------------------------------------- attention
def attn_fwd(q, k, v, cu_q, cu_k, scale, causal=False, quant_p=True, tile_n=128,
             lazy_thr=0.0, p_scale=0):
    """Forward on dequantized operands [tokens, H, D] -> (O float64, lse [H, tokens]).

    p_scale=1: every P block takes the constant exponent ceil(lazy_thr) - 8."""
    lib = _load()
    q, k, v = (_c(a, np.float64) for a in (q, k, v))
    tq, H, D = q.shape
    cq, n = _seg(tq, cu_q)
    ck, _ = _seg(k.shape[0], cu_k)
    o = np.zeros_like(q)
    lse = np.zeros((H, tq), np.float64)
    lib.mxo_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck), n, H, D,
                     float(scale), int(causal), int(quant_p), int(tile_n),
                     float(lazy_thr), _ptr(o), _ptr(lse), tq, int(p_scale))
    return o, lse


def attn_bwd(q, k, v, do, o_bf, do_bf, lse, cu_q, cu_k, scale, causal=False,
             quant_p=True, quant_ds=True, p_scale=0):
    """Backward on dequantized operands -> (dQ, dK, dV) float64 [tokens, H, D].

    do enters dP; do_bf enters Delta = rowsum(do_bf * o_bf) (the method passes
    the same dequantized dO for both, see method_bwd).
    p_scale=1: every P^T block takes the constant exponent -8."""
    lib = _load()
    q, k, v, do, o_bf, do_bf = (_c(a, np.float64) for a in (q, k, v, do, o_bf, do_bf))
    lse = _c(lse, np.float64)
    tq, H, D = q.shape
    cq, n = _seg(tq, cu_q)
    ck, _ = _seg(k.shape[0], cu_k)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    lib.mxo_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(o_bf), _ptr(do_bf),
                     _ptr(lse), _ptr(cq), _ptr(ck), n, H, D, float(scale), int(causal),
                     int(quant_p), int(quant_ds), _ptr(dq), _ptr(dk), _ptr(dv), tq, int(p_scale))
    return dq, dk, dv


# --------------------------------------------------- the method, end to end
def method_fwd(q_bf, k_bf, v_bf, cu_q, cu_k, scale, causal=False, quant=True,
               tile_n=128, lazy_thr=0.0, p_scale=0):
    """Quantize Q, K (1x32 along D) and V (32x1 along keys), then attention."""
    if quant:
        q = qdq(q_bf, ROW, cu_q)
        k = qdq(k_bf, ROW, cu_k)
        v = qdq(v_bf, COL, cu_k)
    else:
        q, k, v = q_bf, k_bf, v_bf
    return attn_fwd(q, k, v, cu_q, cu_k, scale, causal, quant, tile_n, lazy_thr, p_scale)


def method_bwd(q_bf, k_bf, v_bf, do_bf, o_bf, lse, cu_q, cu_k, scale, causal=False,
               quant=True, p_scale=0):
    """Square-block Q, K, dO and row-block V, then the five-GEMM backward.

    Delta = rowsum(dO^ * O) takes the same dequantized dO^ that enters
    dP = dO^ V^ (reading: the backward runs on the quantized operands, and
    the identity sum_j P_ij dP_ij = dO_i . O_i that dS = P (dP - Delta)
    relies on holds for one and the same dO)."""
    if quant:
        q = qdq(q_bf, SQ, cu_q)
        k = qdq(k_bf, SQ, cu_k)
        do = qdq(do_bf, SQ, cu_q)
        v = qdq(v_bf, ROW, cu_k)
    else:
        q, k, do, v = q_bf, k_bf, do_bf, v_bf
    return attn_bwd(q, k, v, do, o_bf, do, lse, cu_q, cu_k, scale, causal,
                    quant, quant, p_scale)


# ------------------------------------------ lower-precision element formats
E2M1, E2M3, E3M2 = 0, 1, 2


def fp_decode(fmt: int, codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.mxo_fp_decode(fmt, int(v)) for v in c.ravel()]).reshape(c.shape)


def fp_encode(fmt: int, vals) -> np.ndarray:
    lib = _load()
    v = np.asarray(vals, dtype=np.float64)
    return np.array([lib.mxo_fp_encode(fmt, float(x)) for x in v.ravel()],
                    dtype=np.uint8).reshape(v.shape)


def fp_max(fmt: int) -> float:
    return float(_load().mxo_fp_max(fmt))


def quantize_mx(x2d, fmt: int):
    """MXFP4 / MXFP6: x[rows, cols] -> (codes u8 [rows, cols] unpacked, E8M0 [rows, cols/32])."""
    lib = _load()
    x = _c(x2d, np.float64)
    rows, cols = x.shape
    q = np.zeros((rows, cols), np.uint8)
    sf = np.zeros((rows, cols // 32), np.uint8)
    lib.mxo_quantize_mx(_ptr(x), rows, cols, fmt, _ptr(q), _ptr(sf))
    return q, sf


def dequantize_mx(q, sf, fmt: int) -> np.ndarray:
    vals = fp_decode(fmt, np.arange(256, dtype=np.uint8) & (0x0F if fmt == E2M1 else 0x3F))
    x = vals[np.asarray(q)]
    return x * np.ldexp(1.0, np.repeat(np.asarray(sf, np.int64), 32, axis=1) - 127)


def quantize_nvfp4(x2d):
    """NVFP4: x[rows, cols] -> (E2M1 codes u8 [rows, cols], E4M3 scales [rows, cols/16],
    fp32 tensor scale)."""
    lib = _load()
    x = _c(x2d, np.float64)
    rows, cols = x.shape
    q = np.zeros((rows, cols), np.uint8)
    sf = np.zeros((rows, cols // 16), np.uint8)
    st = lib.mxo_quantize_nvfp4(_ptr(x), rows, cols, _ptr(q), _ptr(sf))
    return q, sf, st


# ------------------------------------------------------- GEMM+Quantize
def gemm_nt(a, b):
    """y = a b^T in fp64 for a [M, K], b [N, K]."""
    lib = _load()
    a = _c(a, np.float64)
    b = _c(b, np.float64)
    M, K = a.shape
    N = b.shape[0]
    y = np.zeros((M, N), np.float64)
    lib.mxo_gemm_nt(_ptr(a), _ptr(b), M, N, K, _ptr(y))
    return y


def method_gemm_quant(a_bf, b_bf):
    """The GEMM+Quantize step: A, B quantized 1x32 along K, Y = A^ B^^T in fp64,
    then Y quantized ROW (1x32 along N) and COL (32x1 along M).
    Returns (Y, (row payload, row scales), (col payload, col scales))."""
    a = dequantize(*quantize(a_bf, ROW), ROW)
    b = dequantize(*quantize(b_bf, ROW), ROW)
    y = gemm_nt(a, b)
    return y, quantize(y, ROW), quantize(y, COL)


# ------------------------------------------------------ RMSNorm+Quantize
def rmsnorm_quant(x_f32, gamma, eps=1e-6, out_mask=7, seg_len=8192, want_y=False):
    """Fused RMSNorm + MX quantization in the kernel's fp32 order.

    Returns a dict with 'row', 'col', 'sq' -> (payload, compact SF) for the
    requested outputs and optionally 'y' (fp32)."""
    lib = _load()
    x = _c(x_f32, np.float32)
    g = _c(gamma, np.float32)
    T, C = x.shape
    cu = np.minimum(np.arange(0, T + seg_len, seg_len, dtype=np.int64), T)
    cu = np.unique(cu).astype(np.int32)
    out = {}
    bufs = [None] * 6
    if out_mask & 1:
        bufs[0] = np.zeros((T, C), np.uint8)
        bufs[1] = np.zeros((T, C // 32), np.uint8)
    if out_mask & 2:
        bufs[2] = np.zeros((T, C), np.uint8)
        bufs[3] = np.zeros((sf_rows(cu, T), C), np.uint8)
    if out_mask & 4:
        bufs[4] = np.zeros((T, C), np.uint8)
        bufs[5] = np.zeros((sf_rows(cu, T), C // 32), np.uint8)
    y = np.zeros((T, C), np.float32) if want_y else None
    lib.mxo_rmsnorm_quant(_ptr(x), _ptr(g), T, C, ctypes.c_float(eps), out_mask,
                          seg_len, *[_ptr(b) for b in bufs], _ptr(y))
    if out_mask & 1:
        out["row"] = (bufs[0], bufs[1])
    if out_mask & 2:
        out["col"] = (bufs[2], bufs[3])
    if out_mask & 4:
        out["sq"] = (bufs[4], bufs[5])
    if want_y:
        out["y"] = y
    return out
