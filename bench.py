#!/usr/bin/env python
"""Benchmark: one MXFP8 block-scaled attention training step on one GB300.

Workload (the LLM-shaped causal self-attention): B=2, H=16, S=8192, D=128,
Q/K/V/dO bf16 ~ N(0,1) from seed 1.  One step is the whole hot path:
quantize Q and K (32x32 and 1x32 along D, one read each) and V (32x1 along
keys and 1x32 along D, one read), packed scales -> forward -> quantize dO
(32x32) -> backward with FP32 dQ reduction.  value = algorithmic PFLOP/s of the step (forward 4*D and backward
10*D FLOPs per unmasked (query, key) pair, S^2/2 pairs per causal head).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mxfa|reference]
  python bench.py --profile-op fwd|bwd|rmsnorm|gemm|quant_row|quant_col|quant_sq|quant_dual_sq|
                   quant_dual_col [--profile-seq S]
                   [--profile-batch B] [--steps K] [--warmup W]

One JSON line on rank 0; at N=1 it also carries "accuracy": the SQNR of the
step's O, dQ, dK, dV against fp64 attention without quantization on one
(batch, head) of the workload.  --profile-op runs W + K launches of one operation
on a causal case (B=--profile-batch, H=16, S=--profile-seq; for rmsnorm the
fused producer's X[32768, 2048] with row and column outputs; for quant_* one
quantization of the benchmark's Q tensor into packed scales) for kernel
profiling, and prints its timing instead of the benchmark line.

Under torchrun (N > 1) every rank runs the same
per-GPU workload (replicas; no collective on the data path) and value is the
sum of all ranks' work over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B, H, S, D = 2, 16, 8192, 128
CAUSAL = True
# DRAM bytes of one mxfa_bwd call at this workload (preparation, main and post
# kernels), from the ncu capture recorded in profiles/attn_bwd_kernel_llm_traffic.md;
# valid while those kernels are unchanged
BWD_CALL_TRAFFIC = 101825280 + 87026944 + 1336138496 + 917195776 + 134224384 + 31139840
SEED = 1
METRIC = "MXFP8 attn fwd+bwd PFLOP/s (1 GB300)"
NOMINAL_FP8_TFLOPS = 4500.0


def attn_flops(b, h, s, d, causal, per_pair):
    pairs = b * h * (s * s / 2 if causal else s * s)
    return per_pair * d * pairs


FWD_FLOPS = attn_flops(B, H, S, D, CAUSAL, 4)
BWD_FLOPS = attn_flops(B, H, S, D, CAUSAL, 10)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="mxfa", choices=["mxfa", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-components", action="store_true")
    p.add_argument("--no-accuracy", action="store_true")
    p.add_argument("--profile-op", choices=["fwd", "bwd", "rmsnorm", "gemm", "quant_dual_sq",
                                            "quant_dual_col", "quant_row", "quant_col",
                                            "quant_sq"], default=None)
    p.add_argument("--profile-seq", type=int, default=4096)
    p.add_argument("--profile-batch", type=int, default=1)
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm
class GpuStep:
    """Preallocated buffers and the hot path as a sequence of C-ABI calls."""

    def __init__(self, torch, mx, dev, qb, kb, vb, dob):
        self.torch, self.mx, self.dev = torch, mx, dev
        to = lambda b: torch.from_numpy(b.view("int16")).view(torch.bfloat16).reshape(B * S, H, D)
        self.host_in = [to(b).pin_memory() for b in (qb, kb, vb, dob)]
        self.q, self.k, self.v, self.do = [t.to(dev) for t in self.host_in]
        self.seqs = mx.Seqs.dense(B, S)
        u8 = dict(dtype=torch.uint8, device=dev)
        pk = lambda blk: torch.empty(self.seqs.ptiles * H * (16 if blk == 2 else 512), **u8)
        self.mx_out = {}
        for name, blk in (("qR", 0), ("kR", 0), ("vC", 1), ("qS", 2), ("kS", 2), ("doS", 2), ("vR", 0)):
            self.mx_out[name] = mx.Mx(torch.empty((B * S, H, D), **u8), None, pk(blk), blk)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.o = torch.empty((B * S, H, D), **bf)
        self.lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = (torch.empty((B * S, H, D), **bf) for _ in range(3))
        self.ws = torch.empty(mx.mxfa_bwd_workspace_size(B * S, B, H, D, 0), **u8)
        self.host_out = [torch.empty((B * S, H, D), dtype=torch.bfloat16).pin_memory()
                         for _ in range(4)]
        self.scale = 1.0 / math.sqrt(D)
        self.launches_per_step = 4 + 1 + 3  # 4 quantization passes, forward, backward (pre, main, post)

    def quant(self, x, name):
        m = self.mx_out[name]
        out = self.mx.MxOut(m.data.data_ptr(), None, m.sf_packed.data_ptr())
        s = self.seqs
        self.mx.mxfa_quantize(x, s.total, H, D, m.blk, None, s.nseq, s.max_len, s.ptiles, out)

    def fwd(self):
        m = self.mx_out
        self.mx.mxfa_fwd(m["qR"].mx_in(), m["kR"].mx_in(), m["vC"].mx_in(), B, S, H, D, self.scale,
                         CAUSAL, self.o, self.lse)

    def bwd(self, dq_mode=0, dq_static=1.0):
        m = self.mx_out
        self.mx.mxfa_bwd(m["qS"].mx_in(), m["kS"].mx_in(), m["vR"].mx_in(), m["doS"].mx_in(), self.o,
                         self.do, self.lse, B, S, H, D, self.scale, CAUSAL, dq_mode, dq_static,
                         self.dq, self.dk, self.dv, self.ws, self.ws.numel())

    def quant_dual(self, x, name, name_row):
        m, r = self.mx_out[name], self.mx_out[name_row]
        s = self.seqs
        self.mx.mxfa_quantize_dual(x, s.total, H, D, m.blk, None, s.nseq, s.max_len, s.ptiles,
                                   self.mx.MxOut(m.data.data_ptr(), None, m.sf_packed.data_ptr()),
                                   self.mx.MxOut(r.data.data_ptr(), None, r.sf_packed.data_ptr()))

    def step(self):
        # Q, K: 32x32 (backward) and 1x32 (forward) from one read each; V: 32x1
        # (forward) and 1x32 (backward) from one read; dO, known only after
        # the forward in training, is quantized 32x32 then
        self.quant_dual(self.q, "qS", "qR")
        self.quant_dual(self.k, "kS", "kR")
        self.quant_dual(self.v, "vC", "vR")
        self.fwd()
        self.quant(self.do, "doS")
        self.bwd()

    def e2e(self, steps):
        """`steps` steps from pinned host inputs to pinned host outputs, every
        step copying its Q, K, V, dO in and its O, dQ, dK, dV out.  Device
        inputs and outputs are double-buffered: the copy-in of step i+1 and
        the copy-out of step i-1 run on their own streams while step i
        computes.  Returns the milliseconds per step, first copy-in to last
        copy-out."""
        torch = self.torch
        names_in, names_out = ("q", "k", "v", "do"), ("o", "lse", "dq", "dk", "dv")
        if not hasattr(self, "_bufs"):
            own = {n: getattr(self, n) for n in names_in + names_out}
            self._bufs = [own, {n: torch.empty_like(t) for n, t in own.items()}]
        s_cmp = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        in_done, cmp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_cmp)
        s_in.wait_event(t0)
        for i in range(steps):
            b, buf = i % 2, self._bufs[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(cmp_done[b])  # step i-2 no longer reads these inputs
                for n, src in zip(names_in, self.host_in):
                    buf[n].copy_(src, non_blocking=True)
                in_done[b].record(s_in)
            s_cmp.wait_event(in_done[b])
            if i >= 2:
                s_cmp.wait_event(out_done[b])  # step i-2's outputs have left the device
            for n in names_in + names_out:
                setattr(self, n, buf[n])
            self.step()
            cmp_done[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[b])
                for dst, n in zip(self.host_out, ("o", "dq", "dk", "dv")):
                    dst.copy_(buf[n], non_blocking=True)
                out_done[b].record(s_out)
        s_cmp.wait_event(out_done[(steps - 1) % 2])
        t1.record(s_cmp)
        torch.cuda.synchronize()
        for n in names_in + names_out:
            setattr(self, n, self._bufs[0][n])
        return t0.elapsed_time(t1) / steps


def host_link_probe(torch, st, iters=10):
    """The host link's ceiling for the end-to-end figure: the same pinned
    host <-> device copies as one end-to-end step (Q, K, V, dO in; O, dQ, dK,
    dV out), both directions at once on their own streams and nothing else on
    the GPU.  Returns (ms per step, GB/s per direction)."""
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    dev_in = [torch.empty_like(t, device=st.dev) for t in st.host_in]
    dev_out = [st.o, st.dq, st.dk, st.dv]
    cur = torch.cuda.current_stream()

    def once():
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        with torch.cuda.stream(s_in):
            for d, h in zip(dev_in, st.host_in):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s_out):
            for h, d in zip(st.host_out, dev_out):
                h.copy_(d, non_blocking=True)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    ms = time_loop(torch, once, iters, 2)
    nbytes = sum(t.numel() * t.element_size() for t in st.host_in)
    return ms, nbytes / ms / 1e6


def time_loop(torch, fn, iters, warmup, flush=None):
    """Mean per-call device time (ms) with CUDA events on the current stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / iters
    tot = 0.0
    for _ in range(iters):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        tot += a.elapsed_time(b)
    return tot / iters


def time_rotating(torch, fns, iters, warmup):
    """Mean per-call device time (ms) of back-to-back calls that cycle through
    fns, each on its own input and output buffers (together far larger than
    L2, so every call reads its input from HBM), with CUDA events around the
    whole loop: no flush and no per-launch event inside the timed region."""
    for f in fns:
        for _ in range(warmup):
            f()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(iters, len(fns))
    a.record()
    for i in range(n):
        fns[i % len(fns)]()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def quant_slots(torch, mx, st, x, blk, dual, k=4):
    """k copies of x with their own MXFP8 outputs (packed scales, as the step
    writes them) and one quantize call per copy."""
    s = st.seqs
    fns, keep = [], []
    for _ in range(k):
        xi = x.clone()
        if dual:
            m, r = mx.quantize_dual(xi, blk, s)
            o1 = mx.MxOut(m.data.data_ptr(), None, m.sf_packed.data_ptr())
            o2 = mx.MxOut(r.data.data_ptr(), None, r.sf_packed.data_ptr())
            fns.append(lambda xi=xi, o1=o1, o2=o2: mx.mxfa_quantize_dual(
                xi, s.total, H, D, blk, None, s.nseq, s.max_len, s.ptiles, o1, o2))
            keep += [xi, m, r]
        else:
            m = mx.quantize(xi, blk, s)
            o1 = mx.MxOut(m.data.data_ptr(), None, m.sf_packed.data_ptr())
            fns.append(lambda xi=xi, o1=o1: mx.mxfa_quantize(
                xi, s.total, H, D, blk, None, s.nseq, s.max_len, s.ptiles, o1))
            keep += [xi, m]
    return fns, keep


def mxfp8_peak(torch, mx, dev, iters=8192):
    """The tensor pipe's dense MXFP8 peak on this GPU: one CTA per SM issuing
    back-to-back block-scaled MMAs (M128 N256 K32) on resident operands."""
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(nsm, dtype=torch.int64, device=dev)
    mx.mxfa_tensor_peak_probe(64, nsm, cyc)  # warm-up
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    mx.mxfa_tensor_peak_probe(iters, nsm, cyc)
    b.record()
    torch.cuda.synchronize()
    assert mx.device_status() == 0, "device status after the peak probe"
    ms = a.elapsed_time(b)
    macs = iters * 4 * 128 * 256 * 32
    c = cyc.double().mean().item()
    return {"tflops": 2.0 * macs * nsm / (ms * 1e-3) / 1e12, "ms": ms, "sms": nsm,
            "mac_per_clk_per_sm": macs / c, "clock_mhz": c / (ms * 1e3),
            "how": f"{nsm} CTAs x {iters * 4} MMAs (M128 N256 K32, E4M3, resident operands), "
                   "CUDA events around the launch"}


def components(torch, mx, st, iters, warmup, bf16_peak, hbm_peak):
    """Per-kernel figures on the same workload, plus the other workloads' rows."""
    from mxfp8_block_scaled_fa_gb300 import inputs
    dev = st.dev
    res = {}
    res["hbm_timing"] = ("quantizers and RMSNorm+Quantize: back-to-back calls cycling over 4 (2 for "
                         "RMSNorm) input/output copies larger than L2 together, CUDA events around "
                         "the loop")
    fp8_peak = 2.0 * bf16_peak
    st.step()
    t_fwd = time_loop(torch, st.fwd, iters, warmup)
    t_bwd = time_loop(torch, st.bwd, iters, warmup)
    t_bwd16 = time_loop(torch, lambda: st.bwd(1, 1.0), iters, warmup)
    # forward that also writes O as MXFP8 (payload + compact and packed ROW scales)
    u8 = dict(dtype=torch.uint8, device=dev)
    omx = [torch.empty((B * S, H, D), **u8), torch.empty((B * S, H * D // 32), **u8),
           torch.empty(st.seqs.ptiles * H * 512, **u8)]
    omx_s = mx.MxOut(*(t.data_ptr() for t in omx))
    m = st.mx_out
    fwd_mxo = lambda: mx.mxfa_fwd_mxo(m["qR"].mx_in(), m["kR"].mx_in(), m["vC"].mx_in(), B, S, H,
                                      D, st.scale, CAUSAL, st.o, st.lse, omx_s)
    t_fwd_mxo = time_loop(torch, fwd_mxo, iters, warmup)
    del omx
    # backward that also writes dQ, dK, dV as MXFP8 (payload + compact and packed ROW scales)
    gmx = [[torch.empty((B * S, H, D), **u8), torch.empty((B * S, H * D // 32), **u8),
            torch.empty(st.seqs.ptiles * H * 512, **u8)] for _ in range(3)]
    gs = [mx.MxOut(*(t.data_ptr() for t in g)) for g in gmx]
    bwd_mxg = lambda: mx.mxfa_bwd_mxg(m["qS"].mx_in(), m["kS"].mx_in(), m["vR"].mx_in(),
                                      m["doS"].mx_in(), st.o, st.do, st.lse, B, S, H, D, st.scale,
                                      CAUSAL, 0, 1.0, st.dq, st.dk, st.dv, st.ws, st.ws.numel(),
                                      *gs)
    t_bwd_mxg = time_loop(torch, bwd_mxg, iters, warmup)
    del gmx
    st.bwd()
    # HBM-bound calls: back to back over 4 input / output copies (> 400 MB, past L2)
    qt = {}
    for key, x, blk, dual in (("q", st.q, mx.ROW, False), ("qs", st.q, mx.SQ, False),
                              ("qc", st.v, mx.COL, False), ("dsq", st.q, mx.SQ, True),
                              ("dcr", st.v, mx.COL, True)):
        fns, keep = quant_slots(torch, mx, st, x, blk, dual)
        qt[key] = time_rotating(torch, fns, iters, warmup)
        del fns, keep
    t_q, t_qs, t_qc, t_dsq, t_dcr = qt["q"], qt["qs"], qt["qc"], qt["dsq"], qt["dcr"]
    n = B * S * H * D
    res["fwd"] = {"ms": t_fwd, "pflops": FWD_FLOPS / t_fwd / 1e12,
                  "frac_of_4.5": FWD_FLOPS / t_fwd / 1e9 / NOMINAL_FP8_TFLOPS}
    res["fwd_mxfp8_o"] = {"ms": t_fwd_mxo, "pflops": FWD_FLOPS / t_fwd_mxo / 1e12,
                          "note": "forward with O also written as MXFP8 (ROW)"}
    res["bwd_mxfp8_grads"] = {"ms": t_bwd_mxg, "pflops": BWD_FLOPS / t_bwd_mxg / 1e12,
                              "note": "fp32-dQ backward with dQ, dK, dV also written as MXFP8 (ROW)"}
    res["bwd_fp32_dq"] = {"ms": t_bwd, "pflops": BWD_FLOPS / t_bwd / 1e12,
                          "frac_of_4.5": BWD_FLOPS / t_bwd / 1e9 / NOMINAL_FP8_TFLOPS}
    res["bwd_fp16_dq"] = {"ms": t_bwd16, "pflops": BWD_FLOPS / t_bwd16 / 1e12,
                          "frac_of_4.5": BWD_FLOPS / t_bwd16 / 1e9 / NOMINAL_FP8_TFLOPS}
    for key, t, sfb in (("quantize_row", t_q, 1 / 32), ("quantize_col", t_qc, 1 / 32),
                        ("quantize_sq", t_qs, 1 / 1024)):
        gbs = n * (2 + 1 + sfb) / t / 1e6
        res[key] = {"ms": t, "GB_s": gbs, "frac_of_hbm": gbs / hbm_peak}
    # one read, two layouts: 2 B in, (1 + 1/1024) + (1 + 1/32) or 2 (1 + 1/32) B out per element
    for key, t, sfb in (("quantize_dual_sq_row", t_dsq, 1 / 1024 + 1 / 32),
                        ("quantize_dual_col_row", t_dcr, 2 / 32)):
        gbs = n * (2 + 2 + sfb) / t / 1e6
        res[key] = {"ms": t, "GB_s": gbs, "frac_of_hbm": gbs / hbm_peak}
    # fused RMSNorm + Quantize (row + column layouts) on X[32768, 2048]
    x, g, _ = inputs.fused_inputs()
    xd = torch.from_numpy(x.view("int16")).view(torch.bfloat16).to(dev)
    gd = torch.from_numpy(g).to(dev)
    outs = mx.rmsnorm_quant(xd, gd, 1e-6, 8192, 16, outputs=("row", "col"))
    structs = {k: mx.MxOut(v.data.data_ptr(), v.sf_compact.data_ptr(), v.sf_packed.data_ptr())
               for k, v in outs.items()}
    rms = lambda: mx.mxfa_rmsnorm_quant(xd, gd, 32768, 2048, 1e-6, 8192, 16, structs["row"],
                                         structs["col"], None)
    # a second copy of X and its outputs: the calls alternate between them
    xd2 = xd.clone()
    outs2 = mx.rmsnorm_quant(xd2, gd, 1e-6, 8192, 16, outputs=("row", "col"))
    s2 = {k: mx.MxOut(v.data.data_ptr(), v.sf_compact.data_ptr(), v.sf_packed.data_ptr())
          for k, v in outs2.items()}
    rms2 = lambda: mx.mxfa_rmsnorm_quant(xd2, gd, 32768, 2048, 1e-6, 8192, 16, s2["row"], s2["col"],
                                          None)
    t_rms = time_rotating(torch, [rms, rms2], iters, warmup)
    del xd2, outs2
    nb = 32768 * 2048 * (2 + 2 * (1 + 1 / 32))
    res["rmsnorm_quant_row_col"] = {"ms": t_rms, "GB_s": nb / t_rms / 1e6,
                                    "frac_of_hbm": nb / t_rms / 1e6 / hbm_peak}
    del xd, outs
    # jagged cross-attention, 64 sequences (varlen forward + backward)
    qb, kb, vb, dob, cu_q, cu_k = inputs.jagged_attn()
    lq, lk = cu_q[1:] - cu_q[:-1], cu_k[1:] - cu_k[:-1]
    sq, sk = mx.Seqs.varlen(lq, dev), mx.Seqs.varlen(lk, dev)
    tq = lambda b: torch.from_numpy(b.view("int16")).view(torch.bfloat16).to(dev)
    Hj = 8
    qR, kR, vC = mx.quantize(tq(qb), 0, sq), mx.quantize(tq(kb), 0, sk), mx.quantize(tq(vb), 1, sk)
    qS, kS, vR = mx.quantize(tq(qb), 2, sq), mx.quantize(tq(kb), 2, sk), mx.quantize(tq(vb), 0, sk)
    do_t = tq(dob)
    doS = mx.quantize(do_t, 2, sq)
    o, lse = mx.attention_fwd(qR, kR, vC, sq, sk, 1 / math.sqrt(D), False)
    out = (o, lse)
    t_jf = time_loop(torch, lambda: mx.attention_fwd(qR, kR, vC, sq, sk, 1 / math.sqrt(D), False,
                                                     out=out), iters, warmup)
    ws = torch.empty(mx.mxfa_bwd_workspace_size(sq.total, sq.nseq, Hj, D, 0), dtype=torch.uint8,
                     device=dev)
    grads = tuple(torch.empty_like(t) for t in (o, o, o))
    grads = (grads[0], torch.empty((sk.total, Hj, D), dtype=torch.bfloat16, device=dev),
             torch.empty((sk.total, Hj, D), dtype=torch.bfloat16, device=dev))
    t_jb = time_loop(torch, lambda: mx.attention_bwd(qS, kS, vR, doS, o, do_t, lse, sq, sk,
                                                     1 / math.sqrt(D), False, ws=ws, out=grads),
                     iters, warmup)
    pairs = float(np.sum(lq.astype(np.float64) * lk)) * Hj
    res["jagged_fwd"] = {"ms": t_jf, "pflops": 4 * D * pairs / t_jf / 1e12}
    res["jagged_bwd"] = {"ms": t_jb, "pflops": 10 * D * pairs / t_jb / 1e12}
    # accuracy on the sequence with the most queries, head 0 (outputs of the last timed calls)
    i = int(np.argmax(lq))
    a0, a1, k0, k1 = int(cu_q[i]), int(cu_q[i + 1]), int(cu_k[i]), int(cu_k[i + 1])
    f = lambda x, r0, r1: inputs.bf16_bits_to_f32(x[r0:r1, 0, :]).astype(np.float64)
    g = lambda t, r0, r1: t[r0:r1, 0, :].float().cpu().numpy()
    ref = exact_attention(torch, f(qb, a0, a1), f(kb, k0, k1), f(vb, k0, k1), f(dob, a0, a1),
                          1 / math.sqrt(D), False)
    res["jagged_bwd"]["sqnr_db"] = sqnr_db([g(o, a0, a1), g(grads[0], a0, a1), g(grads[1], k0, k1),
                                            g(grads[2], k0, k1)], ref)
    res["jagged_bwd"]["sqnr_sample"] = f"sequence {i} ({a1 - a0} queries x {k1 - k0} keys), head 0"
    del qR, kR, vC, qS, kS, vR, do_t, doS, o, lse, out, ws, grads
    # the outlier workload: B8 H32 S4096 non-causal, outlier recipe on Q and K
    Bo, Ho, So = 8, 32, 4096
    qb, kb, vb, dob = inputs.dense_attn(Bo, Ho, So, D, seed=2, outliers=True)
    so = mx.Seqs.dense(Bo, So)
    to = lambda b: torch.from_numpy(b.view("int16")).view(torch.bfloat16).reshape(Bo * So, Ho, D).to(dev)
    qo, ko, vo, doo = to(qb), to(kb), to(vb), to(dob)
    samp = [inputs.bf16_bits_to_f32(x[0, :, 0, :]).astype(np.float64) for x in (qb, kb, vb, dob)]
    del qb, kb, vb, dob
    fq = [mx.quantize(qo, 0, so), mx.quantize(ko, 0, so), mx.quantize(vo, 1, so)]
    bq = [mx.quantize(qo, 2, so), mx.quantize(ko, 2, so), mx.quantize(vo, 0, so),
          mx.quantize(doo, 2, so)]
    oo, lo = mx.attention_fwd(*fq, so, so, 1 / math.sqrt(D), False)
    t_of = time_loop(torch, lambda: mx.attention_fwd(*fq, so, so, 1 / math.sqrt(D), False,
                                                     out=(oo, lo)), iters, warmup)
    wso = torch.empty(mx.mxfa_bwd_workspace_size(Bo * So, Bo, Ho, D, 0), dtype=torch.uint8, device=dev)
    go = tuple(torch.empty_like(oo) for _ in range(3))
    t_ob = time_loop(torch, lambda: mx.attention_bwd(*bq, oo, doo, lo, so, so, 1 / math.sqrt(D),
                                                     False, ws=wso, out=go), iters, warmup)
    of = attn_flops(Bo, Ho, So, D, False, 4)
    res["outlier_fwd"] = {"ms": t_of, "pflops": of / t_of / 1e12,
                          "workload": "B8 H32 S4096 D128 non-causal, outlier recipe"}
    res["outlier_bwd"] = {"ms": t_ob, "pflops": 2.5 * of / t_ob / 1e12}
    ref = exact_attention(torch, *samp, 1 / math.sqrt(D), False)
    g = lambda t: t[:So, 0, :].float().cpu().numpy()
    res["outlier_bwd"]["sqnr_db"] = sqnr_db([g(oo)] + [g(t) for t in go], ref)
    res["outlier_bwd"]["sqnr_sample"] = "(batch 0, head 0), outputs of the last timed calls"
    del qo, ko, vo, doo, fq, bq, oo, lo, wso, go
    # the forward's rescale threshold and the constant P scale mode on the LLM workload
    sweep = {}
    for thr in (0.0, 4.0, 8.0):
        opts = mx.AttnOpts(thr, mx.P_SCALE_BLOCK)
        t = time_loop(torch, lambda: mx.mxfa_fwd_opts(m["qR"].mx_in(), m["kR"].mx_in(),
                                                      m["vC"].mx_in(), B, S, H, D, st.scale, CAUSAL,
                                                      opts, st.o, st.lse), iters, warmup)
        sweep[f"thr_{thr:g}"] = {"ms": t, "pflops": FWD_FLOPS / t / 1e12}
    res["fwd_rescale_threshold_sweep"] = sweep
    copts = mx.AttnOpts(8.0, mx.P_SCALE_CONST)
    t_fc = time_loop(torch, lambda: mx.mxfa_fwd_opts(m["qR"].mx_in(), m["kR"].mx_in(),
                                                     m["vC"].mx_in(), B, S, H, D, st.scale, CAUSAL,
                                                     copts, st.o, st.lse), iters, warmup)
    t_bc = time_loop(torch, lambda: mx.mxfa_bwd_opts(m["qS"].mx_in(), m["kS"].mx_in(),
                                                     m["vR"].mx_in(), m["doS"].mx_in(), st.o, st.do,
                                                     st.lse, B, S, H, D, st.scale, CAUSAL, copts, 0,
                                                     1.0, st.dq, st.dk, st.dv, st.ws, st.ws.numel()),
                     iters, warmup)
    res["constant_p_scale"] = {"fwd": {"ms": t_fc, "pflops": FWD_FLOPS / t_fc / 1e12},
                               "bwd": {"ms": t_bc, "pflops": BWD_FLOPS / t_bc / 1e12}}
    st.fwd()
    st.bwd()
    # long-key batches: jagged / uniform keys up to 16384 behind 1024 queries, and causal
    # jagged self-attention (16 sequences, H8)
    for kind in ("jagged", "uniform", "causal"):
        qb, kb, vb, dob, cu_q, cu_k, causal = inputs.long_kv_attn(kind)
        lq, lk = cu_q[1:] - cu_q[:-1], cu_k[1:] - cu_k[:-1]
        sq, sk = mx.Seqs.varlen(lq, dev), mx.Seqs.varlen(lk, dev)
        tq = lambda b: torch.from_numpy(b.view("int16")).view(torch.bfloat16).to(dev)
        Hl = 8
        qR, kR, vC = mx.quantize(tq(qb), 0, sq), mx.quantize(tq(kb), 0, sk), mx.quantize(tq(vb), 1, sk)
        qS, kS, vR = mx.quantize(tq(qb), 2, sq), mx.quantize(tq(kb), 2, sk), mx.quantize(tq(vb), 0, sk)
        do_t = tq(dob)
        doS = mx.quantize(do_t, 2, sq)
        o, lse = mx.attention_fwd(qR, kR, vC, sq, sk, 1 / math.sqrt(D), causal)
        out = (o, lse)
        t_f = time_loop(torch, lambda: mx.attention_fwd(qR, kR, vC, sq, sk, 1 / math.sqrt(D), causal,
                                                        out=out), iters, warmup)
        ws = torch.empty(mx.mxfa_bwd_workspace_size(sq.total, sq.nseq, Hl, D, 0), dtype=torch.uint8,
                         device=dev)
        grads = (torch.empty_like(o), torch.empty((sk.total, Hl, D), dtype=torch.bfloat16, device=dev),
                 torch.empty((sk.total, Hl, D), dtype=torch.bfloat16, device=dev))
        t_b = time_loop(torch, lambda: mx.attention_bwd(qS, kS, vR, doS, o, do_t, lse, sq, sk,
                                                        1 / math.sqrt(D), causal, ws=ws, out=grads),
                        iters, warmup)
        pairs = float(np.sum(lq.astype(np.float64) * lk)) * Hl
        if causal:
            pairs = float(np.sum(lq.astype(np.float64) * lq / 2)) * Hl
        res[f"long_kv_{kind}_fwd"] = {"ms": t_f, "pflops": 4 * D * pairs / t_f / 1e12,
                                      "workload": f"16 seqs H8 D128, {kind} keys up to 16384"
                                                  + (", causal" if causal else ", 1024 queries each")}
        res[f"long_kv_{kind}_bwd"] = {"ms": t_b, "pflops": 10 * D * pairs / t_b / 1e12}
        del qR, kR, vC, qS, kS, vR, do_t, doS, o, lse, out, ws, grads
    # GEMM+Quantize: the fused workload's QKV projection, X[32768, 2048] (MXFP8 ROW) x
    # W[6144, 2048] -> Y[32768, 6144] as MXFP8 ROW (Q, K) and COL (V) layouts
    Mg, Kg, Ng = 32768, 2048, 6144
    xg = torch.from_numpy(inputs.normal_bf16((Mg, Kg // 128, 128), 21).view("int16")).view(
        torch.bfloat16).to(dev)
    wg = torch.from_numpy(inputs.normal_bf16((Ng, Kg // 128, 128), 22).view("int16")).view(
        torch.bfloat16).to(dev)
    ag = mx.quantize(xg, 0, mx.Seqs.dense(1, Mg))
    bg = mx.quantize(wg, 0, mx.Seqs.dense(1, Ng))
    del xg, wg
    outs_g = mx.gemm_quant(ag, bg, bf16=False)
    ro, co = outs_g["row"], outs_g["col"]
    so = [mx.MxOut(t.data.data_ptr(), t.sf_compact.data_ptr(), t.sf_packed.data_ptr()) for t in (ro, co)]
    yb = torch.empty((Mg, Ng), dtype=torch.bfloat16, device=dev)
    gfl = 2.0 * Mg * Ng * Kg
    t_gq = time_loop(torch, lambda: mx.mxfa_gemm_quant(ag.mx_in(), bg.mx_in(), Mg, Ng, Kg, None, so[0],
                                                       so[1]), iters, warmup)
    t_gb = time_loop(torch, lambda: mx.mxfa_gemm_quant(ag.mx_in(), bg.mx_in(), Mg, Ng, Kg, yb, None,
                                                       None), iters, warmup)
    res["gemm_quant"] = {"ms": t_gq, "pflops": gfl / t_gq / 1e12,
                         "workload": "X[32768,2048] x W[6144,2048]^T -> Y MXFP8 ROW + COL (packed)",
                         "bf16_out_ms": t_gb, "bf16_out_pflops": gfl / t_gb / 1e12}
    del ag, bg, outs_g, ro, co, yb
    step_q = 2 * t_dsq + t_dcr + t_qs
    res["step_share"] = {"fwd": t_fwd, "bwd": t_bwd, "quantize_4_passes": step_q}
    torch.cuda.synchronize()
    return res


import numpy as np  # noqa: E402  (used by components)


# ------------------------------------------------------------ CPU oracle legs
def oracle_sample(qb, kb, vb, dob, s_len, n_heads):
    """Causal s_len-token prefix of n_heads (batch, head) pairs as one oracle call."""
    from mxfp8_block_scaled_fa_gb300 import inputs
    pairs = [(i // H, i % H) for i in range(min(n_heads, B * H))]
    take = lambda x: np.stack([inputs.bf16_bits_to_f32(x[b, :s_len, h, :]) for b, h in pairs],
                              axis=1).astype(np.float64)
    return take(qb), take(kb), take(vb), take(dob), len(pairs)


def run_oracle_step(oracle, q, k, v, do, scale):
    o, lse = oracle.method_fwd(q, k, v, None, None, scale, True, True, 128, 8.0)
    o_bf = np.asarray(o, np.float32).astype(np.float64)
    oracle.method_bwd(q, k, v, do, o_bf, lse, None, None, scale, True, True)


def cpu_baseline(qb, kb, vb, dob, s_len=4096):
    import oracle
    cores = oracle.num_threads()
    q, k, v, do, n = oracle_sample(qb, kb, vb, dob, s_len, cores)
    scale = 1.0 / math.sqrt(D)
    t0 = time.perf_counter()
    o, lse = oracle.method_fwd(q, k, v, None, None, scale, True, True, 128, 8.0)
    t1 = time.perf_counter()
    o_bf = np.asarray(o, np.float32).astype(np.float64)
    oracle.method_bwd(q, k, v, do, o_bf, lse, None, None, scale, True, True)
    t2 = time.perf_counter()
    dt = t2 - t0
    pairs = (s_len * s_len / 2) * n
    # the tiny workload (B1 H2 S256, non-causal) on one host thread, forward + backward
    from mxfp8_block_scaled_fa_gb300 import inputs
    tq, tk, tv, tdo = (inputs.bf16_bits_to_f32(x).astype(np.float64).reshape(256, 2, D)
                       for x in inputs.dense_attn(1, 2, 256, D, seed=0))
    oracle.set_num_threads(1)
    try:
        u0 = time.perf_counter()
        to, tl = oracle.method_fwd(tq, tk, tv, None, None, scale, False, True, 128, 8.0)
        u1 = time.perf_counter()
        oracle.method_bwd(tq, tk, tv, tdo, np.asarray(to, np.float32).astype(np.float64), tl, None,
                          None, scale, False, True)
        u2 = time.perf_counter()
    finally:
        oracle.set_num_threads(cores)
    tiny_pairs = 2 * 256 * 256
    return {"value": 14 * D * pairs / dt / 1e15, "unit": "PFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"fwd+bwd (quantize, forward, backward) of the causal {s_len}-token prefix of "
                      f"{n} (batch, head) pairs of the workload, heads in parallel, {dt:.1f} s",
            "seconds": dt,
            "fwd": {"seconds": t1 - t0, "PFLOP/s": 4 * D * pairs / (t1 - t0) / 1e15},
            "bwd": {"seconds": t2 - t1, "PFLOP/s": 10 * D * pairs / (t2 - t1) / 1e15},
            "tiny_1_thread": {"workload": "B1 H2 S256 D128 non-causal", "cores": 1,
                              "fwd_seconds": u1 - u0, "bwd_seconds": u2 - u1,
                              "PFLOP/s": 14 * D * tiny_pairs / (u2 - u0) / 1e15}}


def exact_attention(torch, q, k, v, do, scale, causal, chunk=1024):
    """fp64 attention without quantization on the host, for one (sequence,
    head): O = softmax(scale Q K^T) V and its gradients dQ, dK, dV (dS =
    P * (dP - rowsum(dO * O))), in chunks of query rows.  A measurement
    reference for the SQNR figures, independent of the GPU path."""
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    q, k, v, do = f(q), f(k), f(v), f(do)
    lq, lk = q.shape[0], k.shape[0]
    o = torch.empty_like(q)
    dq = torch.empty_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    for r0 in range(0, lq, chunk):
        r1 = min(lq, r0 + chunk)
        s = (q[r0:r1] @ k.T) * scale
        if causal:  # query i sees keys j <= i (queries and keys aligned at 0)
            qi = torch.arange(r0, r1).unsqueeze(1)
            s = s.masked_fill(torch.arange(lk).unsqueeze(0) > qi, float("-inf"))
        p = torch.softmax(s, dim=1)
        oc = p @ v
        o[r0:r1] = oc
        dp = do[r0:r1] @ v.T
        delta = (do[r0:r1] * oc).sum(dim=1, keepdim=True)
        ds = p * (dp - delta)
        dq[r0:r1] = (ds @ k) * scale
        dk += (ds.T @ q[r0:r1]) * scale
        dv += p.T @ do[r0:r1]
    return [t.numpy() for t in (o, dq, dk, dv)]


def sqnr_db(got, ref):
    """Signal-to-quantization-noise ratio (dB) of each output against the reference."""
    out = {}
    for n, g, r in zip(("O", "dQ", "dK", "dV"), got, ref):
        if g is None:
            continue
        g = np.asarray(g, np.float64).reshape(r.shape)
        out[n] = float(10 * np.log10(np.sum(r * r) / max(np.sum((g - r) ** 2), 1e-300)))
    return out


def accuracy(torch, st, qb, kb, vb, dob, b=1, h=5):
    """Error of the GPU step's outputs against fp64 attention without any
    quantization, on one (batch, head) of the workload: SQNR in dB of O, dQ,
    dK and dV, with FP32 dQ (the step) and with FP16 (static scale) dQ."""
    from mxfp8_block_scaled_fa_gb300 import inputs
    take = lambda x: inputs.bf16_bits_to_f32(x[b, :, h, :]).astype(np.float64)
    ref = exact_attention(torch, take(qb), take(kb), take(vb), take(dob), 1.0 / math.sqrt(D), CAUSAL)
    pick = lambda t: t.view(B, S, H, D)[b, :, h, :].float().cpu().numpy()
    res = {"sample": f"(batch {b}, head {h}) of the workload",
           "reference": "fp64 attention without quantization (host, torch fp64)",
           "sqnr_db": sqnr_db([pick(t) for t in (st.o, st.dq, st.dk, st.dv)], ref)}
    st.bwd(1, 1.0)
    torch.cuda.synchronize()
    res["sqnr_db_fp16_dq"] = sqnr_db([None, pick(st.dq), pick(st.dk), pick(st.dv)], ref)
    st.bwd()
    torch.cuda.synchronize()
    return res


def reference_arm(args):
    """The CPU oracle as the reference implementation, on host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from mxfp8_block_scaled_fa_gb300 import inputs
    qb, kb, vb, dob = inputs.dense_attn(B, H, S, D, seed=SEED)
    cores = oracle.num_threads()
    s_len = 2048
    q, k, v, do, n = oracle_sample(qb, kb, vb, dob, s_len, cores)
    scale = 1.0 / math.sqrt(D)
    for _ in range(args.warmup):
        run_oracle_step(oracle, q, k, v, do, scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle_step(oracle, q, k, v, do, scale)
    dt = (time.perf_counter() - t0) / args.steps
    flops = 14 * D * (s_len * s_len / 2) * n
    val = flops / dt / 1e15
    sample = (f"per step: quantize + forward + backward of the causal {s_len}-token prefix of {n} "
              f"(batch, head) pairs of the workload")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "PFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "llm-causal B2 H16 S8192 D128 fwd+bwd", "B": B, "H": H,
                       "seq_len": S, "D": D, "causal": CAUSAL, "seed": SEED},
            "cpu_baseline": {"value": val, "unit": "PFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "PFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def profile_op(args):
    """W + K launches of one operation (B=--profile-batch, H=16, S=--profile-seq, causal)."""
    import torch
    from mxfp8_block_scaled_fa_gb300 import build, inputs
    build.build()
    from mxfp8_block_scaled_fa_gb300 import mxfa
    if args.profile_op == "rmsnorm":
        x, g, _ = inputs.fused_inputs()
        dev = torch.device("cuda", 0)
        xd = torch.from_numpy(x.view("int16")).view(torch.bfloat16).to(dev)
        gd = torch.from_numpy(g).to(dev)
        outs = mxfa.rmsnorm_quant(xd, gd, 1e-6, 8192, 16, outputs=("row", "col"))
        st = {k: mxfa.MxOut(v.data.data_ptr(), v.sf_compact.data_ptr(), v.sf_packed.data_ptr())
              for k, v in outs.items()}
        run = lambda: mxfa.mxfa_rmsnorm_quant(xd, gd, 32768, 2048, 1e-6, 8192, 16, st["row"],
                                               st["col"], None, None)
        ms = time_loop(torch, run, args.steps, args.warmup)
        assert mxfa.device_status() == 0, "device status"
        nb = 32768 * 2048 * (2 + 2 * (1 + 1 / 32))
        print(json.dumps({"profile_op": "rmsnorm", "T": 32768, "C": 2048, "outputs": "row+col",
                          "ms": ms, "GB_s": nb / ms / 1e6}), flush=True)
        return 0
    b, s = args.profile_batch, args.profile_seq
    if args.profile_op == "gemm":
        # the fused workload's QKV projection: X[32768, 2048] x W[6144, 2048]^T, MXFP8 ROW + COL out
        dev = torch.device("cuda", 0)
        Mg, Kg, Ng = 32768, 2048, 6144
        mk = lambda rows, seed: mxfa.quantize(torch.from_numpy(inputs.normal_bf16(
            (rows, Kg // 128, 128), seed).view("int16")).view(torch.bfloat16).to(dev), mxfa.ROW,
            mxfa.Seqs.dense(1, rows))
        ag, bg = mk(Mg, 21), mk(Ng, 22)
        res = mxfa.gemm_quant(ag, bg, bf16=False)
        so = [mxfa.MxOut(res[n].data.data_ptr(), res[n].sf_compact.data_ptr(),
                         res[n].sf_packed.data_ptr()) for n in ("row", "col")]
        run = lambda: mxfa.mxfa_gemm_quant(ag.mx_in(), bg.mx_in(), Mg, Ng, Kg, None, so[0], so[1])
        ms = time_loop(torch, run, args.steps, args.warmup)
        assert mxfa.device_status() == 0, "device status"
        print(json.dumps({"profile_op": "gemm", "M": Mg, "N": Ng, "K": Kg, "ms": ms,
                          "pflops": 2.0 * Mg * Ng * Kg / ms / 1e12}), flush=True)
        return 0
    if args.profile_op.startswith("quant"):
        blk = {"quant_row": 0, "quant_col": 1, "quant_sq": 2, "quant_dual_sq": 2,
               "quant_dual_col": 1}[args.profile_op]
        dual = args.profile_op.startswith("quant_dual")
        qb = inputs.normal_bf16((B, S, H, D), SEED)
        dev = torch.device("cuda", 0)
        q = torch.from_numpy(qb.view("int16")).view(torch.bfloat16).reshape(B * S, H, D).to(dev)
        seqs = mxfa.Seqs.dense(B, S)
        if dual:
            m, r = mxfa.quantize_dual(q, blk, seqs)
            o1 = mxfa.MxOut(m.data.data_ptr(), None, m.sf_packed.data_ptr())
            o2 = mxfa.MxOut(r.data.data_ptr(), None, r.sf_packed.data_ptr())
            run = lambda: mxfa.mxfa_quantize_dual(q, seqs.total, H, D, blk, None, seqs.nseq,
                                                  seqs.max_len, seqs.ptiles, o1, o2)
        else:
            m = mxfa.quantize(q, blk, seqs)
            out = mxfa.MxOut(m.data.data_ptr(), None, m.sf_packed.data_ptr())
            run = lambda: mxfa.mxfa_quantize(q, seqs.total, H, D, blk, None, seqs.nseq, seqs.max_len,
                                             seqs.ptiles, out)
        ms = time_loop(torch, run, args.steps, args.warmup)
        assert mxfa.device_status() == 0, "device status"
        n = B * S * H * D
        nb = n * (2 + 1 + (1 / 1024 if blk == 2 else 1 / 32) + ((1 + 1 / 32) if dual else 0))
        print(json.dumps({"profile_op": args.profile_op, "shape": [B * S, H, D], "ms": ms,
                          "GB_s": nb / ms / 1e6}), flush=True)
        return 0
    qb, kb, vb, dob = inputs.dense_attn(b, H, s, D, seed=SEED)
    dev = torch.device("cuda", 0)
    t = lambda x: torch.from_numpy(x.view("int16")).view(torch.bfloat16).reshape(b * s, H, D).to(dev)
    q, k, v, do = t(qb), t(kb), t(vb), t(dob)
    seqs = mxfa.Seqs.dense(b, s)
    scale = 1.0 / math.sqrt(D)
    qR, kR, vC = mxfa.quantize(q, 0, seqs), mxfa.quantize(k, 0, seqs), mxfa.quantize(v, 1, seqs)
    o, lse = mxfa.attention_fwd(qR, kR, vC, seqs, seqs, scale, CAUSAL)
    if args.profile_op == "fwd":
        run = lambda: mxfa.attention_fwd(qR, kR, vC, seqs, seqs, scale, CAUSAL, out=(o, lse))
        per_pair = 4
    else:
        ops = (mxfa.quantize(q, 2, seqs), mxfa.quantize(k, 2, seqs), mxfa.quantize(v, 0, seqs),
               mxfa.quantize(do, 2, seqs))
        ws = torch.empty(mxfa.mxfa_bwd_workspace_size(b * s, b, H, D, 0), dtype=torch.uint8,
                         device=dev)
        grads = tuple(torch.empty_like(o) for _ in range(3))
        run = lambda: mxfa.attention_bwd(*ops, o, do, lse, seqs, seqs, scale, CAUSAL, ws=ws,
                                         out=grads)
        per_pair = 10
    ms = time_loop(torch, run, args.steps, args.warmup)
    assert mxfa.device_status() == 0, "device status"
    fl = attn_flops(b, H, s, D, CAUSAL, per_pair)
    print(json.dumps({"profile_op": args.profile_op, "B": b, "H": H, "seq_len": s, "D": D,
                      "causal": CAUSAL, "ms": ms, "pflops": fl / ms / 1e12}), flush=True)
    return 0


# ------------------------------------------------------------------ ranks
def slowest_rank(torch, dist, times_ms, device):
    """The largest of each per-rank time over all ranks (every rank gets it)."""
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_pflops(flops_per_rank, world, ms):
    """Whole-job throughput: the work of all ranks over the slowest rank's step time."""
    return flops_per_rank * world / (ms * 1e-3) / 1e15


# ------------------------------------------------------------------ main
def main():
    args = parse()
    if args.impl == "reference":
        return reference_arm(args)
    if args.profile_op:
        return profile_op(args)
    import torch
    import torch.distributed as dist
    from mxfp8_block_scaled_fa_gb300 import build, inputs
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    from mxfp8_block_scaled_fa_gb300 import mxfa
    bf16_peak, hbm_peak, peak_src = load_peaks()
    fp8_peak = 2.0 * bf16_peak
    probe = mxfp8_peak(torch, mxfa, dev)

    qb, kb, vb, dob = inputs.dense_attn(B, H, S, D, seed=SEED)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(qb, kb, vb, dob)
    st = GpuStep(torch, mxfa, dev, qb, kb, vb, dob)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        st.step()
    assert mxfa.device_status() == 0, "device status after warm-up"
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        st.step()
    e1.record()
    barrier()
    ms = e0.elapsed_time(e1) / args.steps
    # the same step repeated for about a second right after the timed region,
    # so that the clock sampler (one sample per 200 ms) sees the GPU under load
    n_sus = max(1, int(math.ceil(1000.0 / max(ms, 1e-3))))
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(n_sus):
        st.step()
    s1.record()
    barrier()
    clk = clocks.stop()
    clk["window"] = (f"timed {args.steps} steps and {n_sus} more steps right after them "
                     f"(about 1 s)")
    ms_sus = s0.elapsed_time(s1) / n_sus
    # end to end through the same C-ABI calls, host buffers in and out
    st.e2e(2)
    barrier()
    ms_e2e = st.e2e(args.steps)
    barrier()
    ms_link, link_gbs = host_link_probe(torch, st)
    barrier()
    if world > 1:
        ms, ms_e2e = slowest_rank(torch, dist, [ms, ms_e2e], dev)
    assert mxfa.device_status() == 0, "device status after timing"
    acc = None
    if rank == 0 and world == 1 and not args.no_accuracy:
        torch.cuda.synchronize()
        acc = accuracy(torch, st, qb, kb, vb, dob)
    comp = None
    if not args.no_components:
        comp = components(torch, mxfa, st, args.steps, args.warmup, bf16_peak, hbm_peak)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    flops = (FWD_FLOPS + BWD_FLOPS) * world
    value = job_pflops(FWD_FLOPS + BWD_FLOPS, world, ms)
    bytes_io = B * S * H * D * 2 * 4
    line = {"metric": METRIC, "value": value, "unit": "PFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": "llm-causal B2 H16 S8192 D128 fwd+bwd (fp32 dQ)", "B": B,
                       "H": H, "seq_len": S, "D": D, "causal": CAUSAL, "seed": SEED,
                       "flops_per_step": FWD_FLOPS + BWD_FLOPS,
                       "l2": "inputs 268 MB (bf16 Q, K, V, dO) > 129 MB L2; no flush",
                       "parallelism": f"replicas x{world}"},
            "frac_of_nominal_4.5": value / world * 1e3 / NOMINAL_FP8_TFLOPS,
            "e2e": {"value": flops / (ms_e2e * 1e-3) / 1e15, "unit": "PFLOP/s",
                    "ms_per_step": ms_e2e, "h2d_bytes_per_step": bytes_io,
                    "overlap": "copy-in of step i+1 and copy-out of step i-1 on their own "
                               "streams during step i (double-buffered device tensors)",
                    "d2h_bytes_per_step": bytes_io,
                    "host_link": {"ms_per_step": ms_link, "GB_s_per_direction": link_gbs,
                                  "frac": ms_link / ms_e2e,
                                  "how": "the same pinned copies in and out of one step, both "
                                         "directions at once, nothing else on the GPU"}},
            "gpu_launches": st.launches_per_step * args.steps,
            "clocks": clk,
            "sustained": {"steps": n_sus, "ms_per_step": ms_sus,
                          "value": job_pflops(FWD_FLOPS + BWD_FLOPS, world, ms_sus),
                          "unit": "PFLOP/s"}}
    if comp is not None:
        sh = comp["step_share"]
        dom = "bwd" if sh["bwd"] >= sh["fwd"] else "fwd"
        t_dom = sh[dom]
        fl = BWD_FLOPS if dom == "bwd" else FWD_FLOPS
        achieved = fl / (t_dom * 1e-3) / 1e12
        line["roofline"] = {"bound": "tensor", "kernel": "attn_bwd_kernel (mxfa_bwd call incl. "
                            "pre/post)" if dom == "bwd" else "attn_fwd_kernel",
                            "achieved": achieved, "peak": probe["tflops"], "unit": "TFLOP/s",
                            "frac": achieved / probe["tflops"],
                            "traffic": BWD_CALL_TRAFFIC if dom == "bwd" else None,
                            "traffic_unit": "bytes per call",
                            "traffic_note": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of "
                                             "bwd_prep_kernel + attn_bwd_kernel + bwd_post_kernel "
                                             "in one capture of this workload "
                                             "(profiles/attn_bwd_kernel_llm_traffic.md), not "
                                             "measured in this run" if dom == "bwd" else
                                             "no capture of this kernel at this workload"),
                            "peak_source": "measured in this run: the dense MXFP8 tensor-pipe "
                                           "peak (mxfa_tensor_peak_probe, see mxfp8_peak)",
                            "peak_probe": probe,
                            "frac_of_bf16x2": achieved / fp8_peak,
                            "bf16x2_source": f"{peak_src} bf16 burst {bf16_peak} x 2 (nominal "
                                             f"fp8/bf16 ratio)",
                            "frac_of_nominal_4500": achieved / NOMINAL_FP8_TFLOPS}
        line["components"] = comp
    if cpu is not None:
        line["cpu_baseline"] = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample",
                                                     "fwd", "bwd", "tiny_1_thread")}
    if acc is not None:
        line["accuracy"] = acc
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
