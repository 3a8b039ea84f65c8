"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching a device (CPU only)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfa.h")


@pytest.fixture(scope="module")
def lib():
    from mxfp8_block_scaled_fa_gb300 import build, mxfa
    build.build()
    return mxfa.lib()


def declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(mxfa_[a-z0-9_]+)\s*\(", txt)))


def test_exports_every_declared_symbol(lib):
    names = declared()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n


def test_no_oracle_in_the_product_library(lib):
    # the product library carries none of the oracle's symbols
    for n in ("mxo_quantize", "mxo_attn_fwd", "mxo_attn_bwd", "mxo_rmsnorm_quant"):
        with pytest.raises(AttributeError):
            getattr(lib, n)


def test_status_strings(lib):
    for s in range(8):
        assert lib.mxfa_status_string(s)
    assert lib.mxfa_version() == 1


def test_packed_tiles_and_sizes(lib):
    from mxfp8_block_scaled_fa_gb300 import mxfa
    assert mxfa.mxfa_packed_tiles(None, 2, 8192) == 128
    assert mxfa.mxfa_packed_tiles(None, 1, 1) == 1
    cu = np.array([0, 5, 133, 133 + 256], np.int32)
    assert mxfa.mxfa_packed_tiles(cu, 3, 0) == 1 + 1 + 2
    assert lib.mxfa_sf_packed_bytes(0, 10, 4) == 10 * 4 * 512
    assert lib.mxfa_sf_packed_bytes(2, 10, 4) == 10 * 4 * 16
    ws = mxfa.mxfa_bwd_workspace_size(1000, 3, 8, 128, 0)
    assert ws >= (16 + 3) * 8 * 2560 + 1000 * 8 * 128 * 4
    assert mxfa.mxfa_bwd_workspace_size(1000, 3, 8, 128, 1) < ws
    assert mxfa.mxfa_bwd_workspace_size(1000, 0, 8, 128, 0) == 0


def _out(data=0x1000, sfc=0x2000, sfp=0x3000):
    from mxfp8_block_scaled_fa_gb300 import mxfa
    return mxfa.MxOut(data, sfc, sfp)


def test_quantize_argument_checks(lib):
    q = lib.mxfa_quantize
    o = _out()
    ref = ctypes.byref
    assert q(None, 256, 2, 128, 0, None, 1, 256, 2, ref(o), None) == 1       # null x
    assert q(0x1000, 256, 2, 64, 0, None, 1, 256, 2, ref(o), None) == 2      # D != 128
    assert q(0x1000, 256, 2, 128, 7, None, 1, 256, 2, ref(o), None) == 1     # bad block kind
    assert q(0x1001, 256, 2, 128, 0, None, 1, 256, 2, ref(o), None) == 3     # misaligned
    assert q(0x1000, 255, 2, 128, 0, None, 1, 256, 2, ref(o), None) == 1     # tokens != nseq*len
    assert q(0x1000, 256, 2, 128, 0, None, 1, 256, 0, ref(o), None) == 1     # packed w/o tiles


def test_sf_unpack_argument_checks(lib):
    u = lib.mxfa_sf_unpack
    assert u(None, 256, 2, 128, 0, None, 1, 256, 2, 0x2000, None) == 1      # null packed
    assert u(0x3000, 256, 2, 128, 0, None, 1, 256, 2, None, None) == 1      # null compact
    assert u(0x3000, 256, 2, 64, 0, None, 1, 256, 2, 0x2000, None) == 2     # D != 128
    assert u(0x3000, 256, 2, 128, 5, None, 1, 256, 2, 0x2000, None) == 1    # bad block kind
    assert u(0x3000, 256, 2, 128, 0, None, 1, 256, 0, 0x2000, None) == 1    # no packed tiles
    assert u(0x3000, 255, 2, 128, 0, None, 1, 256, 2, 0x2000, None) == 1    # tokens != nseq*len


def test_quantize_dual_argument_checks(lib):
    q = lib.mxfa_quantize_dual
    o, o2 = _out(), _out(data=0x4000)
    ref = ctypes.byref
    assert q(0x1000, 256, 2, 128, 0, None, 1, 256, 2, ref(o), ref(o2), None) == 1    # ROW first
    assert q(0x1000, 256, 2, 128, 1, None, 1, 256, 2, ref(o), None, None) == 1       # no ROW output
    assert q(0x1000, 256, 2, 64, 2, None, 1, 256, 2, ref(o), ref(o2), None) == 2     # D != 128
    assert q(0x1000, 256, 2, 128, 2, None, 1, 256, 2, ref(o), ref(_out(data=0x4004)), None) == 3


def test_noalloc_argument_checks(lib):
    # the no-allocation backward validates like mxfa_bwd before it looks at
    # the size of its scratch array or touches a device
    from mxfp8_block_scaled_fa_gb300 import mxfa
    m = mxfa.MxIn(0x1000, 0x2000)
    bad = mxfa.MxIn(0x1000, 0x2004)
    r = ctypes.byref
    n = lib.mxfa_bwd_noalloc
    args = lambda qm, D, o, B=2, S=8192: (r(qm), r(m), r(m), r(m), o, 0x5000, 0x6000, B, S, 16, D,
                                           0.088, 1, 0, 1.0, 0x7000, 0x8000, 0x9000, None)
    assert n(*args(m, 64, 0x4000)) == 2            # D != 128 before the size check
    assert n(*args(m, 128, None)) == 1             # null O
    assert n(*args(bad, 128, 0x4000)) == 3         # misaligned scales
    assert n(*args(m, 128, 0x4000)) == 4           # ~129 MiB of workspace: beyond the array
    assert n(*args(m, 128, 0x4000, B=0)) == 1      # empty batch


def test_lowp_argument_checks(lib):
    f = lib.mxfa_quantize_lowp
    assert f(0x1000, 128, 128, 4, 0, 0x2000, 0x3000, None, None, None) == 1      # format
    assert f(0x1000, 128, 128, 0, 2, 0x2000, 0x3000, None, None, None) == 1      # q layout
    assert f(0x1000, 128, 128, 3, 1, 0x2000, 0x3000, None, 0x4000, None) == 2    # NVFP4 has no MMA form
    assert f(0x1000, 128, 48, 0, 0, 0x2000, 0x3000, None, None, None) == 2       # cols % 32
    assert f(0x1000, 128, 128, 3, 0, 0x2000, 0x3000, None, None, None) == 1      # NVFP4 tensor scale
    assert f(0x1000, 100, 128, 0, 1, 0x2000, 0x3000, 0x5000, None, None) == 2    # atoms need rows % 128
    assert f(0x1008, 128, 128, 0, 1, 0x2000, 0x3000, None, None, None) == 3      # x misaligned
    from mxfp8_block_scaled_fa_gb300 import mxfa
    m = mxfa.MxIn(0x1000, 0x2000)
    g = lib.mxfa_gemm_quant_fmt
    r = ctypes.byref
    assert g(r(m), 4, r(m), 0, 128, 128, 128, 0x4000, None, None, None) == 1     # element format
    assert g(r(m), 3, r(m), 1, 128, 128, 96, 0x4000, None, None, None) == 2      # K % 128


def test_attention_options_checks(lib):
    # the *_opts calls validate their options before any launch
    from mxfp8_block_scaled_fa_gb300 import mxfa
    m = mxfa.MxIn(0x1000, 0x2000)
    r = ctypes.byref
    f = lib.mxfa_fwd_opts
    fargs = lambda o: (r(m), r(m), r(m), 1, 256, 2, 128, 0.1, 0, o, 0x4000, 0x5000, None)
    assert f(*fargs(r(mxfa.AttnOpts(-1.0, 0)))) == 1       # threshold below 0
    assert f(*fargs(r(mxfa.AttnOpts(8.5, 0)))) == 1        # threshold above 8
    assert f(*fargs(r(mxfa.AttnOpts(float("nan"), 0)))) == 1
    assert f(*fargs(r(mxfa.AttnOpts(4.0, 2)))) == 1        # unknown P scale mode
    assert f(*fargs(r(mxfa.AttnOpts(4.0, 1)))[:6] + (96,) + fargs(None)[7:]) == 2   # D
    b = lib.mxfa_bwd_opts
    ws = mxfa.mxfa_bwd_workspace_size(256, 1, 2, 128, 0)
    bargs = lambda o, wsb=ws: (r(m), r(m), r(m), r(m), 0x4000, 0x5000, 0x6000, 1, 256, 2, 128, 0.1,
                               0, o, 0, 1.0, 0x7000, 0x8000, 0x9000, 0xA000, wsb, None)
    assert b(*bargs(r(mxfa.AttnOpts(8.0, 3)))) == 1
    assert b(*bargs(r(mxfa.AttnOpts(8.0, 1)), ws - 1)) == 4  # workspace still checked
    vf = lib.mxfa_varlen_fwd_opts
    assert vf(r(m), r(m), r(m), None, None, 2, 10, 10, 20, 20, 2, 2, 2, 128, 0.1, 0, None, 0x4000,
              0x5000, None) == 1                            # varlen needs cu_seqlens


def test_attention_argument_checks(lib):
    from mxfp8_block_scaled_fa_gb300 import mxfa
    m = mxfa.MxIn(0x1000, 0x2000)
    bad = mxfa.MxIn(0x1008, 0x2000)
    r = ctypes.byref
    f = lib.mxfa_fwd
    assert f(r(m), r(m), r(m), 1, 256, 2, 96, 0.1, 0, 0x4000, 0x5000, None) == 2   # D
    assert f(r(bad), r(m), r(m), 1, 256, 2, 128, 0.1, 0, 0x4000, 0x5000, None) == 3
    assert f(r(m), r(m), r(m), 0, 256, 2, 128, 0.1, 0, 0x4000, 0x5000, None) == 1   # B
    assert f(r(m), r(m), r(m), 1, 256, 2, 128, -1.0, 0, 0x4000, 0x5000, None) == 1  # scale
    assert f(None, r(m), r(m), 1, 256, 2, 128, 0.1, 0, 0x4000, 0x5000, None) == 1
    b = lib.mxfa_bwd
    ws = mxfa.mxfa_bwd_workspace_size(256, 1, 2, 128, 0)
    args = lambda mode, st, wsb: (r(m), r(m), r(m), r(m), 0x4000, 0x5000, 0x6000, 1, 256, 2, 128,
                                  0.1, 0, mode, st, 0x7000, 0x8000, 0x9000, 0xA000, wsb, None)
    assert b(*args(0, 1.0, ws - 1)) == 4           # workspace too small
    assert b(*args(2, 1.0, ws)) == 1               # bad dq mode
    assert b(*args(1, 3.0, ws)) == 1               # static scale not a power of two
    v = lib.mxfa_varlen_fwd
    assert v(r(m), r(m), r(m), None, None, 2, 10, 10, 20, 20, 2, 2, 2, 128, 0.1, 0, 0x4000,
             0x5000, None) == 1                    # varlen needs cu_seqlens


def test_rmsnorm_argument_checks(lib):
    o = _out(sfp=None)
    r = ctypes.byref
    f = lib.mxfa_rmsnorm_quant
    assert f(0x1000, 0x2000, 64, 300, 1e-6, 64, 2, r(o), None, None, None) == 2    # C
    assert f(0x1000, 0x2000, 64, 256, 1e-6, 48, 2, r(o), None, None, None) == 2    # seg_len
    assert f(0x1000, 0x2000, 64, 256, 1e-6, 64, 2, None, None, None, None) == 1    # no output
    assert f(0x1000, 0x2000, 64, 256, 1e-6, 64, 4, r(o), None, None, None) == 2    # C != H*128


def test_mxfp8_output_argument_checks(lib):
    # the calls with MXFP8 outputs validate those outputs before any launch
    from mxfp8_block_scaled_fa_gb300 import mxfa
    m = mxfa.MxIn(0x1000, 0x2000)
    r = ctypes.byref
    f = lib.mxfa_fwd_mxo
    fargs = lambda omx, D=128: (r(m), r(m), r(m), 1, 256, 2, D, 0.1, 0, 0x4000, 0x5000, omx, None)
    assert f(*fargs(None)) == 1                                  # o_mx required
    assert f(*fargs(r(_out(data=None)))) == 1                    # o_mx->data required
    assert f(*fargs(r(_out(data=0x1008)))) == 3                  # payload not 16-byte aligned
    assert f(*fargs(r(_out(sfc=0x2001)))) == 3                   # compact scales not 4-byte aligned
    assert f(*fargs(r(_out(sfp=0x3004)))) == 3                   # packed scales not 16-byte aligned
    assert f(*fargs(r(_out()), D=96)) == 2                       # D still checked
    v = lib.mxfa_varlen_fwd_mxo
    assert v(r(m), r(m), r(m), None, None, 2, 10, 10, 20, 20, 2, 2, 2, 128, 0.1, 0, 0x4000, 0x5000,
             r(_out()), None) == 1                               # varlen needs cu_seqlens
    b = lib.mxfa_bwd_mxg
    ws = mxfa.mxfa_bwd_workspace_size(256, 1, 2, 128, 0)
    bargs = lambda dq, dk, dv, wsb=ws: (r(m), r(m), r(m), r(m), 0x4000, 0x5000, 0x6000, 1, 256, 2,
                                        128, 0.1, 0, 0, 1.0, 0x7000, 0x8000, 0x9000, 0xA000, wsb,
                                        dq, dk, dv, None)
    assert b(*bargs(r(_out(sfc=None)), None, None)) == 1         # dQ packed scales need compact
    assert b(*bargs(None, r(_out(data=0x1004)), None)) == 3      # dK payload misaligned
    assert b(*bargs(None, None, r(_out(data=None)))) == 1        # dV payload required
    assert b(*bargs(None, None, None, ws - 1)) == 4              # workspace still checked
    vb = lib.mxfa_varlen_bwd_mxg
    assert vb(r(m), r(m), r(m), r(m), 0x4000, 0x5000, 0x6000, None, None, 2, 10, 10, 20, 20, 2, 2,
              2, 128, 0.1, 0, 0, 1.0, 0x7000, 0x8000, 0x9000, 0xA000, ws, None, None, None,
              None) == 1                                         # varlen needs cu_seqlens


def test_package_exposes_the_public_api():
    # the package forwards the binding's public names without loading the library
    import mxfp8_block_scaled_fa_gb300 as pkg
    for n in ("Mx", "MxIn", "MxOut", "Seqs", "ROW", "COL", "SQ", "quantize", "sf_pack", "sf_unpack",
              "attention_fwd", "attention_bwd", "rmsnorm_quant", "device_status", "lib",
              "MxfaError", "mxfa_fwd", "mxfa_bwd", "mxfa_fwd_mxo", "mxfa_bwd_mxg"):
        assert getattr(pkg, n) is not None, n
