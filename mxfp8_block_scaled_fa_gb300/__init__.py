"""mxfa -- MXFP8 block-scaled FlashAttention (forward + backward) for GB300.

The compute path is the C-ABI library ``libmxfa.so`` (hand-written CUDA for
sm_103a); :mod:`.mxfa` is a thin ctypes binding over it whose functions carry
the C names (``mxfa_quantize``, ``mxfa_fwd``, ``mxfa_bwd``, ...).  PyTorch is
used only for device memory and streams.  There is no CPU fallback: every
call fails loudly when the library is missing.
"""
from . import inputs  # noqa: F401  (seeded synthetic workloads; no arithmetic)


def __getattr__(name):
    if name.startswith("mxfa_") or name in ("lib", "MxfaError",
                                            "Mx", "MxIn", "MxOut", "Seqs", "ROW", "COL", "SQ",
                                            "AttnOpts", "P_SCALE_BLOCK", "P_SCALE_CONST",
                                            "RESCALE_THRESHOLD",
                                            "quantize", "quantize_dual", "sf_pack", "sf_unpack", "attention_fwd",
                                            "attention_bwd", "rmsnorm_quant", "gemm_quant", "quantize_lowp",
                                            "LOWP_MXFP4", "LOWP_MXFP6_E2M3", "LOWP_MXFP6_E3M2",
                                            "LOWP_NVFP4", "LOWP_CODES", "LOWP_MMA", "ELEM_E4M3", "ELEM_E2M3", "ELEM_E3M2",
                                            "ELEM_E2M1",
                                            "device_status"):
        from . import mxfa as _m
        return getattr(_m, name)
    raise AttributeError(name)
