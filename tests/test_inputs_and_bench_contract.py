"""CPU checks of the seeded workload generators (the shapes, counts and
ranges the configurations prescribe) and of the benchmark's JSON contract on
its reference arm (the oracle on host cores)."""
import json
import os
import subprocess
import sys

import numpy as np

from mxfp8_block_scaled_fa_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_outlier_recipe_counts():
    # 1% of the (head, d) channels of Q and K scaled by 20, then 0.1% of the
    # elements by 200; V untouched unless outliers_v; the base values are the
    # same draws as without outliers
    B, H, S, D = 2, 4, 256, 128
    base = inputs.dense_attn(B, H, S, D, seed=5)
    out = inputs.dense_attn(B, H, S, D, seed=5, outliers=True)
    f = lambda b: inputs.bf16_bits_to_f32(b).astype(np.float64)
    n_ch, n_el = round(0.01 * H * D), round(0.001 * B * S * H * D)
    for t in (0, 1):
        a, b = f(base[t]), f(out[t])
        nz = np.abs(a) > 1e-3
        ratio = np.where(nz, b / np.where(nz, a, 1.0), 1.0)
        # channels: columns where most elements carry the x20 factor
        col_scaled = (np.abs(ratio.reshape(B * S, H * D) / 20.0 - 1) < 0.02).mean(axis=0) > 0.9
        assert col_scaled.sum() == n_ch
        # elements: about n_el carry an extra x200 (x4000 on a scaled channel)
        big = (np.abs(ratio / 200.0 - 1) < 0.02) | (np.abs(ratio / 4000.0 - 1) < 0.02)
        assert abs(int(big.sum()) - n_el) <= n_el // 50 + 2
    np.testing.assert_array_equal(base[2], out[2])   # V
    np.testing.assert_array_equal(base[3], out[3])   # dO


def test_jagged_lengths_and_packing():
    qb, kb, vb, dob, cu_q, cu_k = inputs.jagged_attn()
    lq, lk = np.diff(cu_q), np.diff(cu_k)
    assert len(lq) == len(lk) == 64
    assert lq.min() >= 64 and lq.max() <= 2048 and lk.min() >= 32 and lk.max() <= 1024
    assert qb.shape == (cu_q[-1], 8, 128) and dob.shape == qb.shape
    assert kb.shape == (cu_k[-1], 8, 128) and vb.shape == kb.shape
    # seeded: the same call gives the same lengths
    assert np.array_equal(inputs.jagged_attn()[4], cu_q)


def test_fused_inputs_ranges():
    x, g, do = inputs.fused_inputs(T=256, C=256, B=1, S=256, H=2, seed=4)
    assert x.shape == (256, 256) and do.shape == (1, 256, 2, 128)
    assert g.dtype == np.float32 and g.min() >= 0.5 and g.max() <= 1.5


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
