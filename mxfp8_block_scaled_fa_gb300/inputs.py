"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the attention method: only random numbers
(numpy ``Generator(PCG64(seed))``), float32 -> bf16 round-to-nearest-even and
the shapes of the workloads.  Both the CUDA path and the CPU oracle consume
the exact same bf16 bytes produced here.

Recipes (tensor order Q, K, V, dO; every tensor float32 ``standard_normal``
rounded to bf16 unless stated):

* ``tiny``      B=1 H=2 S=256 D=128, non-causal, seed 0
* ``llm``       B=2 H=16 S=8192 D=128, causal, seed 1
* ``outliers``  B=8 H=32 S=4096 D=128, non-causal, seed 2; after the four
  normal draws, Q then K each get 1% of their H*D channels (``choice`` without
  replacement) scaled by 20 and then 0.1% of their elements scaled by 200;
  variant ``outliers_v`` also scales 0.1% of V's elements by 200
* ``jagged``    64 sequences, query lengths ``integers(64, 2048, endpoint)``
  then key lengths ``integers(32, 1024, endpoint)``, H=8 D=128, non-causal,
  packed token-major with ``cu_seqlens``, seed 3
* ``fused``     X[32768, 2048] normal, gamma ``uniform(0.5, 1.5)`` float32,
  dO[4, 8192, 16, 128] normal, eps 1e-6, attention causal, seed 4
* ``long_kv``   long-key jagged batches (key lengths up to 16384), H=8 D=128,
  16 sequences, seed 5: ``jagged`` cross-attention with 1024 queries per
  sequence and key lengths ``integers(1024, 16384, endpoint)``;
  ``uniform`` the same with every key length 16384; ``causal`` self-attention
  with lengths ``integers(1024, 16384, endpoint)``, causal
"""
from __future__ import annotations

import numpy as np

CONFIGS = {
    "tiny": dict(B=1, H=2, S=256, D=128, causal=False, seed=0),
    "llm": dict(B=2, H=16, S=8192, D=128, causal=True, seed=1),
    "outliers": dict(B=8, H=32, S=4096, D=128, causal=False, seed=2),
    "jagged": dict(nseq=64, H=8, D=128, causal=False, seed=3,
                   lq=(64, 2048), lk=(32, 1024)),
    "fused": dict(T=32768, C=2048, B=4, S=8192, H=16, D=128, causal=True, seed=4,
                  eps=1e-6),
    "long_kv": dict(nseq=16, H=8, D=128, seed=5, lq_cross=1024, lk=(1024, 16384)),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    # finite patterns are <= 0xFF7FFFFF, so adding at most 0x8000 cannot wrap
    t = (b >> 16) & 1
    t += b
    t += 0x7FFF
    r = (t >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng, shape):
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def dense_attn(B, H, S, D, seed, outliers=False, outliers_v=False):
    """Q, K, V, dO as bf16 bits [B, S, H, D] (uint16)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (B, S, H, D)
    f = [rng.standard_normal(shape, dtype=np.float32) for _ in range(4)]
    if outliers:
        n_ch = int(round(0.01 * H * D))
        n_el = int(round(0.001 * B * S * H * D))
        for t in (f[0], f[1]):
            ch = rng.choice(H * D, size=n_ch, replace=False)
            t.reshape(B * S, H * D)[:, ch] *= np.float32(20.0)
            el = rng.choice(t.size, size=n_el, replace=False)
            t.reshape(-1)[el] *= np.float32(200.0)
        if outliers_v:
            el = rng.choice(f[2].size, size=n_el, replace=False)
            f[2].reshape(-1)[el] *= np.float32(200.0)
    return tuple(f32_to_bf16_bits(t) for t in f)


def jagged_lengths(nseq, lq, lk, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    sq = rng.integers(lq[0], lq[1], size=nseq, endpoint=True)
    sk = rng.integers(lk[0], lk[1], size=nseq, endpoint=True)
    return rng, sq.astype(np.int64), sk.astype(np.int64)


def varlen_attn(lens_q, lens_k, H, D, seed, rng=None):
    """Packed Q, dO [total_q, H, D], K, V [total_k, H, D] bf16 bits + cu_seqlens."""
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    lens_q = np.asarray(lens_q, np.int64)
    lens_k = np.asarray(lens_k, np.int64)
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    q = _normal_bf16(rng, (tq, H, D))
    k = _normal_bf16(rng, (tk, H, D))
    v = _normal_bf16(rng, (tk, H, D))
    do = _normal_bf16(rng, (tq, H, D))
    return q, k, v, do, cu_q, cu_k


def jagged_attn(nseq=64, H=8, D=128, seed=3, lq=(64, 2048), lk=(32, 1024)):
    rng, sq, sk = jagged_lengths(nseq, lq, lk, seed)
    return varlen_attn(sq, sk, H, D, seed, rng=rng)


def fused_inputs(T=32768, C=2048, B=4, S=8192, H=16, D=128, seed=4):
    """X bf16 bits [T, C], gamma float32 [C], dO bf16 bits [B, S, H, D]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = _normal_bf16(rng, (T, C))
    gamma = rng.uniform(0.5, 1.5, size=C).astype(np.float32)
    do = _normal_bf16(rng, (B, S, H, D))
    return x, gamma, do


def normal_bf16(shape, seed):
    """Generic seeded N(0,1) bf16 bits of any shape."""
    return _normal_bf16(np.random.Generator(np.random.PCG64(seed)), shape)


def long_kv_lengths(kind, nseq=16, seed=5, lq_cross=1024, lk=(1024, 16384)):
    """(query lengths, key lengths, causal) of a long-key batch: kind is
    'jagged' (cross, jagged keys), 'uniform' (cross, every key length lk[1])
    or 'causal' (self-attention, jagged lengths)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(lk[0], lk[1], size=nseq, endpoint=True).astype(np.int64)
    if kind == "jagged":
        return np.full(nseq, lq_cross, np.int64), lens, False
    if kind == "uniform":
        return np.full(nseq, lq_cross, np.int64), np.full(nseq, lk[1], np.int64), False
    if kind == "causal":
        return lens, lens.copy(), True
    raise ValueError(kind)


def long_kv_attn(kind, nseq=16, H=8, D=128, seed=5):
    """Q, K, V, dO bf16 bits (packed token-major) + cu_seqlens + causal flag."""
    lq, lk, causal = long_kv_lengths(kind, nseq, seed)
    q, k, v, do, cu_q, cu_k = varlen_attn(lq, lk, H, D, seed + 100)
    return q, k, v, do, cu_q, cu_k, causal
