"""Test-side helpers: host/device transfer, packed-scale decoding, metrics.

The packed-scale decoder below is written from the layout stated in
include/mxfa.h, independently of the kernels, so that the kernels' packed
output can be compared with the oracle's compact scales.
"""
from __future__ import annotations

import numpy as np

from mxfp8_block_scaled_fa_gb300 import inputs


def to_dev(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def f64(bits: np.ndarray) -> np.ndarray:
    return inputs.bf16_bits_to_f32(bits).astype(np.float64)


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def seq_lengths(cu):
    cu = np.asarray(cu, np.int64)
    return cu[1:] - cu[:-1]


def unpack_packed(packed: np.ndarray, blk: int, lens, H: int, D: int = 128):
    """Packed scales -> (compact scales, padding bytes) for the given lengths."""
    lens = np.asarray(lens, np.int64)
    cols = H * D
    starts = np.concatenate([[0], np.cumsum(lens)])[:-1]
    b32 = np.concatenate([[0], np.cumsum((lens + 31) // 32)])[:-1]
    t128 = np.concatenate([[0], np.cumsum((lens + 127) // 128)])[:-1]
    per = 16 if blk == 2 else 512
    packed = packed.reshape(-1, H, per)
    pads = []
    if blk == 0:
        comp = np.zeros((int(lens.sum()), cols // 32), np.uint8)
        r = np.arange(128)
        kb = np.arange(D // 32)
        off = (r[:, None] % 32) * 16 + (r[:, None] // 32) * 4 + kb[None, :]   # [128, 4]
        for g, L in enumerate(lens):
            for t in range((L + 127) // 128):
                atom = packed[t128[g] + t]          # [H, 512]
                vals = atom[:, off]                 # [H, 128, 4]
                n = min(128, L - t * 128)
                comp[starts[g] + t * 128: starts[g] + t * 128 + n] = \
                    vals[:, :n, :].transpose(1, 0, 2).reshape(n, cols // 32)
                pads.append(vals[:, n:, :].ravel())
    elif blk == 1:
        comp = np.zeros((int(((lens + 31) // 32).sum()), cols), np.uint8)
        d = np.arange(D)
        kb = np.arange(4)
        off = (d[None, :] % 32) * 16 + (d[None, :] // 32) * 4 + kb[:, None]   # [4, 128]
        for g, L in enumerate(lens):
            nb = (L + 31) // 32
            for t in range((L + 127) // 128):
                vals = packed[t128[g] + t][:, off]  # [H, 4, 128]
                m = min(4, nb - t * 4)
                comp[b32[g] + t * 4: b32[g] + t * 4 + m] = \
                    vals[:, :m, :].transpose(1, 0, 2).reshape(m, cols)
                pads.append(vals[:, m:, :].ravel())
    else:
        comp = np.zeros((int(((lens + 31) // 32).sum()), cols // 32), np.uint8)
        for g, L in enumerate(lens):
            nb = (L + 31) // 32
            for t in range((L + 127) // 128):
                vals = packed[t128[g] + t].reshape(H, 4, 4)   # [H, tb, db]
                m = min(4, nb - t * 4)
                comp[b32[g] + t * 4: b32[g] + t * 4 + m] = \
                    vals[:, :m, :].transpose(1, 0, 2).reshape(m, cols // 32)
                pads.append(vals[:, m:, :].ravel())
    pad = np.concatenate(pads) if pads else np.zeros(0, np.uint8)
    return comp, pad


def rel_fro(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def max_abs(got, ref) -> float:
    return float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))))


def sqnr_db(got, ref) -> float:
    ref = np.asarray(ref, np.float64)
    err = np.asarray(got, np.float64) - ref
    return float(10 * np.log10(np.sum(ref * ref) / max(np.sum(err * err), 1e-300)))
