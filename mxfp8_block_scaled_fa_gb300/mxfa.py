"""Thin ctypes binding over libmxfa.so (include/mxfa.h).

The functions named ``mxfa_*`` mirror the C entry points one to one and only
marshal arguments (torch CUDA tensors -> device pointers, the current torch
stream -> ``cudaStream_t``).  The helpers below them (``quantize``,
``attention_fwd`` ...) allocate outputs with torch and call those entry points;
every arithmetic step runs in the library's CUDA kernels.  Nothing here falls
back to the CPU: a missing library or a CUDA-less process raises.

A training step on bf16 q, k, v, do of shape [B * S, H, 128] (dense, causal):

    seqs = Seqs.dense(B, S)
    scale = 1 / math.sqrt(128)
    o, lse = attention_fwd(quantize(q, ROW, seqs), quantize(k, ROW, seqs),
                           quantize(v, COL, seqs), seqs, seqs, scale, causal=True)
    dq, dk, dv = attention_bwd(quantize(q, SQ, seqs), quantize(k, SQ, seqs),
                               quantize(v, ROW, seqs), quantize(do, SQ, seqs),
                               o, do, lse, seqs, seqs, scale, causal=True)

Jagged batches use ``Seqs.varlen(lengths, device)`` for queries and keys;
``o_mx=True`` / ``grads_mx=True`` also return O / the gradients as MXFP8.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from . import build as _build

ROW, COL, SQ = 0, 1, 2
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
           3: "pointer not 16-byte aligned", 4: "workspace too small", 5: "CUDA error",
           6: "device wait timed out", 7: "device index check failed"}


class MxfaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_STATUS.get(status, status)} (status {status})")
        self.status = status


class MxOut(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("sf_compact", ctypes.c_void_p),
                ("sf_packed", ctypes.c_void_p)]


class MxIn(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("sf", ctypes.c_void_p)]


P_SCALE_BLOCK, P_SCALE_CONST = 0, 1
RESCALE_THRESHOLD = 8.0


class AttnOpts(ctypes.Structure):
    """mxfa_attn_opts: forward rescale threshold (log2 units) and the P scale mode."""
    _fields_ = [("rescale_threshold", ctypes.c_float), ("p_scale", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmxfa.so from the package's build folder (raises if absent)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                "libmxfa.so is not built: run mxfp8_block_scaled_fa_gb300.build.build()")
        L = ctypes.CDLL(_build.LIB)
        P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        S = ctypes.c_size_t
        sig = {
            "mxfa_status_string": (ctypes.c_char_p, [I]),
            "mxfa_version": (I, []),
            "mxfa_packed_tiles": (I64, [P, I, I]),
            "mxfa_sf_packed_bytes": (S, [I, I64, I]),
            "mxfa_quantize": (I, [P, I64, I, I, I, P, I, I, I64, P, P]),
            "mxfa_sf_pack": (I, [P, I64, I, I, I, P, I, I, I64, P, P]),
            "mxfa_quantize_dual": (I, [P, I64, I, I, I, P, I, I, I64, P, P, P]),
            "mxfa_sf_unpack": (I, [P, I64, I, I, I, P, I, I, I64, P, P]),
            "mxfa_fwd": (I, [P, P, P, I, I, I, I, F, I, P, P, P]),
            "mxfa_varlen_fwd": (I, [P, P, P, P, P, I, I, I, I64, I64, I64, I64, I, I, F, I, P, P,
                                    P]),
            "mxfa_fwd_mxo": (I, [P, P, P, I, I, I, I, F, I, P, P, P, P]),
            "mxfa_varlen_fwd_mxo": (I, [P, P, P, P, P, I, I, I, I64, I64, I64, I64, I, I, F, I, P,
                                        P, P, P]),
            "mxfa_fwd_opts": (I, [P, P, P, I, I, I, I, F, I, P, P, P, P]),
            "mxfa_varlen_fwd_opts": (I, [P, P, P, P, P, I, I, I, I64, I64, I64, I64, I, I, F, I,
                                         P, P, P, P]),
            "mxfa_bwd_opts": (I, [P, P, P, P, P, P, P, I, I, I, I, F, I, P, I, F, P, P, P, P, S,
                                  P]),
            "mxfa_varlen_bwd_opts": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I64, I64, I64, I64,
                                         I, I, F, I, P, I, F, P, P, P, P, S, P]),
            "mxfa_bwd_workspace_size": (S, [I64, I, I, I, I]),
            "mxfa_bwd": (I, [P, P, P, P, P, P, P, I, I, I, I, F, I, I, F, P, P, P, P, S, P]),
            "mxfa_varlen_bwd": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I64, I64, I64, I64, I, I,
                                    F, I, I, F, P, P, P, P, S, P]),
            "mxfa_bwd_mxg": (I, [P, P, P, P, P, P, P, I, I, I, I, F, I, I, F, P, P, P, P, S, P, P,
                                 P, P]),
            "mxfa_varlen_bwd_mxg": (I, [P, P, P, P, P, P, P, P, P, I, I, I, I64, I64, I64, I64, I,
                                        I, F, I, I, F, P, P, P, P, S, P, P, P, P]),
            "mxfa_rmsnorm_quant": (I, [P, P, I64, I64, F, I, I, P, P, P, P]),
            "mxfa_get_device_status": (I, [P, ctypes.POINTER(ctypes.c_uint)]),
            "mxfa_gemm_quant": (I, [P, P, I64, I64, I64, P, P, P, P]),
            "mxfa_gemm_quant_fmt": (I, [P, I, P, I, I64, I64, I64, P, P, P, P]),
            "mxfa_quantize_lowp": (I, [P, I64, I, I, I, P, P, P, P, P]),
            "mxfa_tensor_peak_probe": (I, [I, I, P, P]),
            "mxfa_bwd_noalloc": (I, [P, P, P, P, P, P, P, I, I, I, I, F, I, I, F, P, P, P, P]),
            "mxfa_bwd_noalloc_scratch_bytes": (S, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(st: int, where: str):
    if st != 0:
        raise MxfaError(st, where)


# ------------------------------------------------------------ C-named calls
def mxfa_packed_tiles(cu_host: Optional[np.ndarray], nseq: int, seqlen: int) -> int:
    if cu_host is None:
        return int(lib().mxfa_packed_tiles(None, nseq, seqlen))
    cu = np.ascontiguousarray(cu_host, dtype=np.int32)
    return int(lib().mxfa_packed_tiles(cu.ctypes.data_as(ctypes.c_void_p), nseq, seqlen))


def mxfa_quantize(x, tokens, H, D, blk, cu_seqlens, nseq, max_seqlen, packed_tiles, out: MxOut,
                  stream=None):
    _check(lib().mxfa_quantize(_p(x), tokens, H, D, blk, _p(cu_seqlens), nseq, max_seqlen,
                               packed_tiles, ctypes.byref(out), _stream(stream)), "mxfa_quantize")


def mxfa_sf_pack(sf_compact, tokens, H, D, blk, cu_seqlens, nseq, max_seqlen, packed_tiles,
                 sf_packed, stream=None):
    _check(lib().mxfa_sf_pack(_p(sf_compact), tokens, H, D, blk, _p(cu_seqlens), nseq, max_seqlen,
                              packed_tiles, _p(sf_packed), _stream(stream)), "mxfa_sf_pack")


def mxfa_sf_unpack(sf_packed, tokens, H, D, blk, cu_seqlens, nseq, max_seqlen, packed_tiles,
                   sf_compact, stream=None):
    _check(lib().mxfa_sf_unpack(_p(sf_packed), tokens, H, D, blk, _p(cu_seqlens), nseq,
                                max_seqlen, packed_tiles, _p(sf_compact), _stream(stream)),
           "mxfa_sf_unpack")


def mxfa_fwd(q: MxIn, k: MxIn, v: MxIn, B, S, H, D, scale, causal, o, lse, stream=None):
    _check(lib().mxfa_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), B, S, H, D,
                          float(scale), int(causal), _p(o), _p(lse), _stream(stream)), "mxfa_fwd")


def mxfa_varlen_fwd(q, k, v, cu_q, cu_k, nseq, max_sq, max_sk, total_q, total_k, ptq, ptk, H, D,
                    scale, causal, o, lse, stream=None):
    _check(lib().mxfa_varlen_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), _p(cu_q),
                                 _p(cu_k), nseq, max_sq, max_sk, total_q, total_k, ptq, ptk, H, D,
                                 float(scale), int(causal), _p(o), _p(lse), _stream(stream)),
           "mxfa_varlen_fwd")


def mxfa_fwd_mxo(q: MxIn, k: MxIn, v: MxIn, B, S, H, D, scale, causal, o, lse, o_mx: MxOut,
                 stream=None):
    _check(lib().mxfa_fwd_mxo(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), B, S, H, D,
                              float(scale), int(causal), _p(o), _p(lse), ctypes.byref(o_mx),
                              _stream(stream)), "mxfa_fwd_mxo")


def mxfa_varlen_fwd_mxo(q, k, v, cu_q, cu_k, nseq, max_sq, max_sk, total_q, total_k, ptq, ptk, H,
                        D, scale, causal, o, lse, o_mx: MxOut, stream=None):
    _check(lib().mxfa_varlen_fwd_mxo(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), _p(cu_q),
                                     _p(cu_k), nseq, max_sq, max_sk, total_q, total_k, ptq, ptk, H,
                                     D, float(scale), int(causal), _p(o), _p(lse),
                                     ctypes.byref(o_mx), _stream(stream)), "mxfa_varlen_fwd_mxo")


def mxfa_bwd_workspace_size(total_q, nseq, H, D, dq_mode) -> int:
    return int(lib().mxfa_bwd_workspace_size(total_q, nseq, H, D, dq_mode))


def mxfa_bwd(q, k, v, do_mx, o, do, lse, B, S, H, D, scale, causal, dq_mode, dq_static, dq, dk,
             dv, ws, ws_bytes, stream=None):
    _check(lib().mxfa_bwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(do_mx),
                          _p(o), _p(do), _p(lse), B, S, H, D, float(scale), int(causal), dq_mode,
                          float(dq_static), _p(dq), _p(dk), _p(dv), _p(ws), ws_bytes,
                          _stream(stream)), "mxfa_bwd")


def mxfa_bwd_noalloc(q, k, v, do_mx, o, do, lse, B, S, H, D, scale, causal, dq_mode, dq_static,
                     dq, dk, dv, stream=None):
    """mxfa_bwd without a caller workspace (the library's built-in scratch array)."""
    _check(lib().mxfa_bwd_noalloc(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                  ctypes.byref(do_mx), _p(o), _p(do), _p(lse), B, S, H, D,
                                  float(scale), int(causal), dq_mode, float(dq_static), _p(dq),
                                  _p(dk), _p(dv), _stream(stream)), "mxfa_bwd_noalloc")


def mxfa_varlen_bwd(q, k, v, do_mx, o, do, lse, cu_q, cu_k, nseq, max_sq, max_sk, total_q,
                    total_k, ptq, ptk, H, D, scale, causal, dq_mode, dq_static, dq, dk, dv, ws,
                    ws_bytes, stream=None):
    _check(lib().mxfa_varlen_bwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                 ctypes.byref(do_mx), _p(o), _p(do), _p(lse), _p(cu_q), _p(cu_k),
                                 nseq, max_sq, max_sk, total_q, total_k, ptq, ptk, H, D,
                                 float(scale), int(causal), dq_mode, float(dq_static), _p(dq),
                                 _p(dk), _p(dv), _p(ws), ws_bytes, _stream(stream)),
           "mxfa_varlen_bwd")


def mxfa_rmsnorm_quant(x, gamma, T, C, eps, seg_len, H, row: Optional[MxOut],
                       col: Optional[MxOut], sq: Optional[MxOut], stream=None):
    ref = lambda m: ctypes.byref(m) if m is not None else None
    _check(lib().mxfa_rmsnorm_quant(_p(x), _p(gamma), T, C, float(eps), seg_len, H, ref(row),
                                    ref(col), ref(sq), _stream(stream)), "mxfa_rmsnorm_quant")


def mxfa_get_device_status(stream=None) -> int:
    flags = ctypes.c_uint(0)
    st = lib().mxfa_get_device_status(_stream(stream), ctypes.byref(flags))
    return st


# ----------------------------------------------------------- convenience layer
@dataclass
class Seqs:
    """Host-side description of packed sequences (dense = uniform lengths)."""
    nseq: int
    max_len: int
    total: int
    cu_host: Optional[np.ndarray]      # int32 [nseq+1] or None (uniform)
    cu_dev: Optional[torch.Tensor]     # int32 device copy or None
    ptiles: int                        # sum ceil(len/128)
    blocks32: int                      # sum ceil(len/32)

    @staticmethod
    def dense(B: int, S: int) -> "Seqs":
        return Seqs(B, S, B * S, None, None, B * math.ceil(S / 128), B * math.ceil(S / 32))

    @staticmethod
    def varlen(lengths: Sequence[int], device) -> "Seqs":
        lens = np.asarray(lengths, dtype=np.int64)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        cu_dev = torch.from_numpy(cu).to(device)
        return Seqs(len(lens), int(lens.max()) if len(lens) else 0, int(cu[-1]), cu, cu_dev,
                    int(np.sum((lens + 127) // 128)), int(np.sum((lens + 31) // 32)))


@dataclass
class Mx:
    """An MXFP8 tensor produced by the library (payload + scales)."""
    data: torch.Tensor                 # uint8 [tokens, H, D]
    sf_compact: Optional[torch.Tensor]
    sf_packed: Optional[torch.Tensor]
    blk: int

    def mx_in(self) -> MxIn:
        return MxIn(self.data.data_ptr(), self.sf_packed.data_ptr())


def _sf_shapes(blk, seqs: Seqs, H, D):
    cols = H * D
    if blk == ROW:
        comp = (seqs.total, cols // 32)
    elif blk == COL:
        comp = (seqs.blocks32, cols)
    else:
        comp = (seqs.blocks32, cols // 32)
    packed = seqs.ptiles * H * (16 if blk == SQ else 512)
    return comp, packed


def quantize(x: torch.Tensor, blk: int, seqs: Seqs, compact=True, packed=True,
             stream=None) -> Mx:
    """bf16 [tokens, H, D] (or [B, S, H, D]) -> Mx via mxfa_quantize."""
    H, D = x.shape[-2], x.shape[-1]
    x3 = x.reshape(-1, H, D)
    dev = x.device
    data = torch.empty(x3.shape, dtype=torch.uint8, device=dev)
    comp_shape, pbytes = _sf_shapes(blk, seqs, H, D)
    sfc = torch.empty(comp_shape, dtype=torch.uint8, device=dev) if compact else None
    sfp = torch.empty(max(pbytes, 16), dtype=torch.uint8, device=dev) if packed else None
    out = MxOut(data.data_ptr(), _p(sfc), _p(sfp))
    mxfa_quantize(x3, seqs.total, H, D, blk, seqs.cu_dev, seqs.nseq, seqs.max_len, seqs.ptiles,
                  out, stream)
    return Mx(data, sfc, sfp, blk)


def mxfa_quantize_dual(x, tokens, H, D, blk, cu_seqlens, nseq, max_seqlen, packed_tiles,
                       out: MxOut, out_row: MxOut, stream=None):
    _check(lib().mxfa_quantize_dual(_p(x), tokens, H, D, blk, _p(cu_seqlens), nseq, max_seqlen,
                                    packed_tiles, ctypes.byref(out), ctypes.byref(out_row),
                                    _stream(stream)), "mxfa_quantize_dual")


def quantize_dual(x: torch.Tensor, blk: int, seqs: Seqs, stream=None):
    """bf16 [tokens, H, D] -> (Mx in layout blk (COL or SQ), Mx in ROW) from one read."""
    H, D = x.shape[-2], x.shape[-1]
    x3 = x.reshape(-1, H, D)
    dev = x.device
    outs, structs = [], []
    for b in (blk, ROW):
        data = torch.empty(x3.shape, dtype=torch.uint8, device=dev)
        comp_shape, pbytes = _sf_shapes(b, seqs, H, D)
        sfc = torch.empty(comp_shape, dtype=torch.uint8, device=dev)
        sfp = torch.empty(max(pbytes, 16), dtype=torch.uint8, device=dev)
        outs.append(Mx(data, sfc, sfp, b))
        structs.append(MxOut(data.data_ptr(), sfc.data_ptr(), sfp.data_ptr()))
    mxfa_quantize_dual(x3, seqs.total, H, D, blk, seqs.cu_dev, seqs.nseq, seqs.max_len, seqs.ptiles,
                       structs[0], structs[1], stream)
    return outs[0], outs[1]


def sf_pack(sf_compact: torch.Tensor, blk: int, seqs: Seqs, H: int, D: int = 128,
            stream=None) -> torch.Tensor:
    _, pbytes = _sf_shapes(blk, seqs, H, D)
    sfp = torch.empty(max(pbytes, 16), dtype=torch.uint8, device=sf_compact.device)
    mxfa_sf_pack(sf_compact, seqs.total, H, D, blk, seqs.cu_dev, seqs.nseq, seqs.max_len,
                 seqs.ptiles, sfp, stream)
    return sfp


def sf_unpack(sf_packed: torch.Tensor, blk: int, seqs: Seqs, H: int, D: int = 128,
              stream=None) -> torch.Tensor:
    """Packed scales -> compact scales (the inverse of sf_pack)."""
    comp_shape, _ = _sf_shapes(blk, seqs, H, D)
    sfc = torch.empty(comp_shape, dtype=torch.uint8, device=sf_packed.device)
    mxfa_sf_unpack(sf_packed, seqs.total, H, D, blk, seqs.cu_dev, seqs.nseq, seqs.max_len,
                   seqs.ptiles, sfc, stream)
    return sfc


def _opts_ref(opts):
    return None if opts is None else ctypes.byref(opts)


def mxfa_fwd_opts(q, k, v, B, S, H, D, scale, causal, opts, o, lse, stream=None):
    _check(lib().mxfa_fwd_opts(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), B, S, H, D,
                               float(scale), int(causal), _opts_ref(opts), _p(o), _p(lse),
                               _stream(stream)), "mxfa_fwd_opts")


def mxfa_varlen_fwd_opts(q, k, v, cu_q, cu_k, nseq, max_sq, max_sk, total_q, total_k, ptq, ptk, H,
                         D, scale, causal, opts, o, lse, stream=None):
    _check(lib().mxfa_varlen_fwd_opts(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), _p(cu_q),
                                      _p(cu_k), nseq, max_sq, max_sk, total_q, total_k, ptq, ptk,
                                      H, D, float(scale), int(causal), _opts_ref(opts), _p(o),
                                      _p(lse), _stream(stream)), "mxfa_varlen_fwd_opts")


def mxfa_bwd_opts(q, k, v, do_mx, o, do, lse, B, S, H, D, scale, causal, opts, dq_mode, dq_static,
                  dq, dk, dv, ws, ws_bytes, stream=None):
    _check(lib().mxfa_bwd_opts(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                               ctypes.byref(do_mx), _p(o), _p(do), _p(lse), B, S, H, D,
                               float(scale), int(causal), _opts_ref(opts), dq_mode,
                               float(dq_static), _p(dq), _p(dk), _p(dv), _p(ws), ws_bytes,
                               _stream(stream)), "mxfa_bwd_opts")


def mxfa_varlen_bwd_opts(q, k, v, do_mx, o, do, lse, cu_q, cu_k, nseq, max_sq, max_sk, total_q,
                         total_k, ptq, ptk, H, D, scale, causal, opts, dq_mode, dq_static, dq, dk,
                         dv, ws, ws_bytes, stream=None):
    _check(lib().mxfa_varlen_bwd_opts(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                      ctypes.byref(do_mx), _p(o), _p(do), _p(lse), _p(cu_q),
                                      _p(cu_k), nseq, max_sq, max_sk, total_q, total_k, ptq, ptk,
                                      H, D, float(scale), int(causal), _opts_ref(opts), dq_mode,
                                      float(dq_static), _p(dq), _p(dk), _p(dv), _p(ws), ws_bytes,
                                      _stream(stream)), "mxfa_varlen_bwd_opts")


def attention_fwd(q: Mx, k: Mx, v: Mx, seqs_q: Seqs, seqs_k: Seqs, scale: float,
                  causal: bool = False, stream=None, out=None, o_mx: bool = False,
                  opts: Optional[AttnOpts] = None):
    """Forward on quantized operands -> (O bf16 [tokens, H, D], lse fp32), and with
    o_mx=True also O as MXFP8 (Mx with ROW compact and packed scales) as a third item.
    opts (AttnOpts) selects the rescale threshold and the P scale mode (no MXFP8 O then)."""
    if opts is not None and o_mx:
        raise ValueError("opts and o_mx cannot be combined")
    H, D = q.data.shape[-2], q.data.shape[-1]
    dev = q.data.device
    o = out[0] if out is not None else torch.empty(q.data.shape, dtype=torch.bfloat16, device=dev)
    omx = omx_s = None
    if o_mx:
        u8 = dict(dtype=torch.uint8, device=dev)
        omx = Mx(torch.empty(q.data.shape, **u8), torch.empty((seqs_q.total, H * D // 32), **u8),
                 torch.empty(seqs_q.ptiles * H * 512, **u8), ROW)
        omx_s = MxOut(omx.data.data_ptr(), omx.sf_compact.data_ptr(), omx.sf_packed.data_ptr())
    if seqs_q.cu_host is None and seqs_k.cu_host is None:
        lse = out[1] if out is not None else torch.empty((seqs_q.nseq, H, seqs_q.max_len),
                                                         dtype=torch.float32, device=dev)
        args = (q.mx_in(), k.mx_in(), v.mx_in(), seqs_q.nseq, seqs_q.max_len, H, D, scale,
                causal, o, lse)
        if o_mx:
            mxfa_fwd_mxo(*args, omx_s, stream)
        elif opts is not None:
            mxfa_fwd_opts(*args[:9], opts, o, lse, stream)
        else:
            mxfa_fwd(*args, stream)
    else:
        lse = out[1] if out is not None else torch.empty((H, seqs_q.total), dtype=torch.float32,
                                                         device=dev)
        args = (q.mx_in(), k.mx_in(), v.mx_in(), seqs_q.cu_dev, seqs_k.cu_dev, seqs_q.nseq,
                seqs_q.max_len, seqs_k.max_len, seqs_q.total, seqs_k.total, seqs_q.ptiles,
                seqs_k.ptiles, H, D, scale, causal, o, lse)
        if o_mx:
            mxfa_varlen_fwd_mxo(*args, omx_s, stream)
        elif opts is not None:
            mxfa_varlen_fwd_opts(*args[:16], opts, o, lse, stream)
        else:
            mxfa_varlen_fwd(*args, stream)
    return (o, lse, omx) if o_mx else (o, lse)


def mxfa_bwd_mxg(q, k, v, do_mx, o, do, lse, B, S, H, D, scale, causal, dq_mode, dq_static, dq,
                 dk, dv, ws, ws_bytes, dq_mx, dk_mx, dv_mx, stream=None):
    ref = lambda m: ctypes.byref(m) if m is not None else None
    _check(lib().mxfa_bwd_mxg(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                              ctypes.byref(do_mx), _p(o), _p(do), _p(lse), B, S, H, D,
                              float(scale), int(causal), dq_mode, float(dq_static), _p(dq), _p(dk),
                              _p(dv), _p(ws), ws_bytes, ref(dq_mx), ref(dk_mx), ref(dv_mx),
                              _stream(stream)), "mxfa_bwd_mxg")


def mxfa_varlen_bwd_mxg(q, k, v, do_mx, o, do, lse, cu_q, cu_k, nseq, max_sq, max_sk, total_q,
                        total_k, ptq, ptk, H, D, scale, causal, dq_mode, dq_static, dq, dk, dv, ws,
                        ws_bytes, dq_mx, dk_mx, dv_mx, stream=None):
    ref = lambda m: ctypes.byref(m) if m is not None else None
    _check(lib().mxfa_varlen_bwd_mxg(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                     ctypes.byref(do_mx), _p(o), _p(do), _p(lse), _p(cu_q),
                                     _p(cu_k), nseq, max_sq, max_sk, total_q, total_k, ptq, ptk, H,
                                     D, float(scale), int(causal), dq_mode, float(dq_static),
                                     _p(dq), _p(dk), _p(dv), _p(ws), ws_bytes, ref(dq_mx),
                                     ref(dk_mx), ref(dv_mx), _stream(stream)),
           "mxfa_varlen_bwd_mxg")


def attention_bwd(q: Mx, k: Mx, v: Mx, do_mx: Mx, o: torch.Tensor, do: torch.Tensor,
                  lse: torch.Tensor, seqs_q: Seqs, seqs_k: Seqs, scale: float,
                  causal: bool = False, dq_mode: int = 0, dq_static: float = 1.0, stream=None,
                  ws=None, out=None, grads_mx: bool = False, opts: Optional[AttnOpts] = None):
    """Backward on quantized operands -> (dQ, dK, dV) bf16; with grads_mx=True also the
    three gradients as MXFP8 (Mx with ROW compact and packed scales), six items in all.
    opts (AttnOpts) selects the P scale mode (no MXFP8 gradients then)."""
    if opts is not None and grads_mx:
        raise ValueError("opts and grads_mx cannot be combined")
    H, D = q.data.shape[-2], q.data.shape[-1]
    dev = q.data.device
    wsb = mxfa_bwd_workspace_size(seqs_q.total, seqs_q.nseq, H, D, dq_mode)
    if ws is None:
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    if out is None:
        dq = torch.empty(q.data.shape, dtype=torch.bfloat16, device=dev)
        dk = torch.empty(k.data.shape, dtype=torch.bfloat16, device=dev)
        dv = torch.empty(v.data.shape, dtype=torch.bfloat16, device=dev)
    else:
        dq, dk, dv = out
    gmx = gs = None
    if grads_mx:
        u8 = dict(dtype=torch.uint8, device=dev)
        gmx = [Mx(torch.empty(t.shape, **u8), torch.empty((sq.total, H * D // 32), **u8),
                  torch.empty(sq.ptiles * H * 512, **u8), ROW)
               for t, sq in ((dq, seqs_q), (dk, seqs_k), (dv, seqs_k))]
        gs = [MxOut(m.data.data_ptr(), m.sf_compact.data_ptr(), m.sf_packed.data_ptr())
              for m in gmx]
    if seqs_q.cu_host is None and seqs_k.cu_host is None:
        args = (q.mx_in(), k.mx_in(), v.mx_in(), do_mx.mx_in(), o, do, lse, seqs_q.nseq,
                seqs_q.max_len, H, D, scale, causal, dq_mode, dq_static, dq, dk, dv, ws,
                ws.numel())
        if grads_mx:
            mxfa_bwd_mxg(*args, *gs, stream)
        elif opts is not None:
            mxfa_bwd_opts(*args[:13], opts, *args[13:], stream)
        else:
            mxfa_bwd(*args, stream)
    else:
        args = (q.mx_in(), k.mx_in(), v.mx_in(), do_mx.mx_in(), o, do, lse, seqs_q.cu_dev,
                seqs_k.cu_dev, seqs_q.nseq, seqs_q.max_len, seqs_k.max_len, seqs_q.total,
                seqs_k.total, seqs_q.ptiles, seqs_k.ptiles, H, D, scale, causal, dq_mode,
                dq_static, dq, dk, dv, ws, ws.numel())
        if grads_mx:
            mxfa_varlen_bwd_mxg(*args, *gs, stream)
        elif opts is not None:
            mxfa_varlen_bwd_opts(*args[:20], opts, *args[20:], stream)
        else:
            mxfa_varlen_bwd(*args, stream)
    return (dq, dk, dv, *gmx) if grads_mx else (dq, dk, dv)


def rmsnorm_quant(x: torch.Tensor, gamma: torch.Tensor, eps: float, seg_len: int, H: int,
                  outputs=("row", "col", "sq"), packed=True, stream=None):
    """Fused RMSNorm + quantization -> dict name -> Mx (compact + packed scales)."""
    T, C = x.shape
    dev = x.device
    seqs = Seqs.dense(T // seg_len, seg_len) if T % seg_len == 0 else None
    res, structs = {}, {}
    for name, blk in (("row", ROW), ("col", COL), ("sq", SQ)):
        if name not in outputs:
            continue
        data = torch.empty((T, C), dtype=torch.uint8, device=dev)
        nb32 = (T + 31) // 32
        comp = {ROW: (T, C // 32), COL: (nb32, C), SQ: (nb32, C // 32)}[blk]
        sfc = torch.empty(comp, dtype=torch.uint8, device=dev)
        sfp = None
        if packed:
            if seqs is None:
                raise ValueError("packed scales need T to be a multiple of seg_len")
            sfp = torch.empty(seqs.ptiles * H * (16 if blk == SQ else 512), dtype=torch.uint8,
                              device=dev)
        res[name] = Mx(data, sfc, sfp, blk)
        structs[name] = MxOut(data.data_ptr(), sfc.data_ptr(), _p(sfp))
    mxfa_rmsnorm_quant(x, gamma, T, C, eps, seg_len, H, structs.get("row"), structs.get("col"),
                       structs.get("sq"), stream)
    return res


def mxfa_gemm_quant(a: MxIn, b: MxIn, M, N, K, y_bf16, y_row: Optional[MxOut],
                    y_col: Optional[MxOut], stream=None):
    ref = lambda m: ctypes.byref(m) if m is not None else None
    _check(lib().mxfa_gemm_quant(ctypes.byref(a), ctypes.byref(b), M, N, K, _p(y_bf16), ref(y_row),
                                 ref(y_col), _stream(stream)), "mxfa_gemm_quant")


LOWP_MXFP4, LOWP_MXFP6_E2M3, LOWP_MXFP6_E3M2, LOWP_NVFP4 = 0, 1, 2, 3
LOWP_CODES, LOWP_MMA = 0, 1
ELEM_E4M3, ELEM_E2M3, ELEM_E3M2, ELEM_E2M1 = 0, 1, 2, 3


def mxfa_quantize_lowp(x, rows, cols, fmt, q_layout, q, sf, sf_packed, tensor_scale, stream=None):
    _check(lib().mxfa_quantize_lowp(_p(x), rows, cols, fmt, q_layout, _p(q), _p(sf), _p(sf_packed),
                                    _p(tensor_scale), _stream(stream)), "mxfa_quantize_lowp")


def quantize_lowp(x: torch.Tensor, fmt: int, packed: bool = False, mma: bool = False, stream=None):
    """bf16 [rows, cols] -> dict: 'q' u8 [rows, cols] (codes one per byte, or with
    mma=True the MMA operand form of the MX formats), 'sf' scales, optional
    'sf_packed' (MX formats), and 'tensor_scale' (NVFP4, a 1-element fp32 tensor)."""
    rows, cols = x.shape[0], x.numel() // x.shape[0]
    dev = x.device
    u8 = dict(dtype=torch.uint8, device=dev)
    q = torch.empty((rows, cols), **u8)
    sf = torch.empty((rows, cols // (16 if fmt == LOWP_NVFP4 else 32)), **u8)
    sfp = torch.empty((rows // 128) * (cols // 128) * 512, **u8) if packed else None
    ts = torch.empty(1, dtype=torch.float32, device=dev) if fmt == LOWP_NVFP4 else None
    mxfa_quantize_lowp(x, rows, cols, fmt, LOWP_MMA if mma else LOWP_CODES, q, sf, sfp, ts, stream)
    return {"q": q, "sf": sf, "sf_packed": sfp, "tensor_scale": ts}


def mxfa_gemm_quant_fmt(a: MxIn, a_fmt, b: MxIn, b_fmt, M, N, K, y_bf16, y_row, y_col, stream=None):
    ref = lambda m: ctypes.byref(m) if m is not None else None
    _check(lib().mxfa_gemm_quant_fmt(ctypes.byref(a), a_fmt, ctypes.byref(b), b_fmt, M, N, K,
                                     _p(y_bf16), ref(y_row), ref(y_col), _stream(stream)),
           "mxfa_gemm_quant_fmt")


def mxfa_tensor_peak_probe(iters, ctas, cycles, stream=None):
    _check(lib().mxfa_tensor_peak_probe(int(iters), int(ctas), _p(cycles), _stream(stream)),
           "mxfa_tensor_peak_probe")


def gemm_quant(a: Mx, b: Mx, bf16: bool = True, row: bool = True, col: bool = True,
               stream=None):
    """Y = A B^T on ROW-quantized A [M, K] and B [N, K] (Mx with packed scales, as
    quantize(x.view(rows, K // 128, 128), ROW, Seqs.dense(1, rows)) makes them) ->
    dict with 'bf16' (tensor [M, N]) and 'row' / 'col' (Mx over [M, N])."""
    M, K = a.data.shape[0], a.data.numel() // a.data.shape[0]
    N = b.data.shape[0]
    dev = a.data.device
    u8 = dict(dtype=torch.uint8, device=dev)
    res, outs = {}, {}
    if bf16:
        res["bf16"] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    for name, blk, comp in (("row", ROW, (M, N // 32)), ("col", COL, (M // 32, N))):
        if (name == "row" and row) or (name == "col" and col):
            m = Mx(torch.empty((M, N), **u8), torch.empty(comp, **u8),
                   torch.empty((M // 128) * (N // 128) * 512, **u8), blk)
            res[name] = m
            outs[name] = MxOut(m.data.data_ptr(), m.sf_compact.data_ptr(), m.sf_packed.data_ptr())
    mxfa_gemm_quant(a.mx_in(), b.mx_in(), M, N, K, res.get("bf16"), outs.get("row"),
                    outs.get("col"), stream)
    return res


def device_status(stream=None) -> int:
    """Synchronise and return (and clear) the kernels' device status (0 = ok)."""
    return mxfa_get_device_status(stream)
