#!/usr/bin/env python3
"""Benchmark of the NVFP4 LoRA-linear hot path on one GB300 (or N replicas).

One step = one forward + input-gradient pass of the Llama-3B-shaped decoder-layer
projection stack (workload "layer-3b": M = 8 x 1024 tokens, hidden 3072,
q/k/v/o 3072 -> 3072/1024/1024/3072, gate|up 3072 -> 2 x 8192, down 8192 -> 3072,
r = 16 LoRA on every projection): both fused RMSNorm -> NVFP4 quantisers, every
activation/gradient quantisation, the fused SiLU-multiply -> NVFP4, the 12 NVFP4
GEMMs with fused LoRA branches, and the RMSNorm and SiLU-multiply backward
kernels.  The attention core and its backward are replaced by seeded tensors.

metric = NVFP4 frozen-projection GEMM FLOPs (2*M*N*K over the 12 GEMMs) divided by
the device time of the whole step (all kernels), in TFLOP/s.  Also reported: layer
tokens/s; the per-step median and an L2-flushed figure; each GEMM kernel's own
TFLOP/s; the memory-bound calls' GB/s (warm and L2-flushed); a sub-line for each
other workload (q-3b, mlp-3b, attn-1b: fwd + input-gradient passes); model tokens/s
projected from the layer stacks (layer-3b x 28, a 1B-shaped stack x 16); the LoRA
adapter gradients; the BF16 comparator; the oracle on the host cores; and the
end-to-end figure through pinned host buffers.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch one process per GPU with torch.distributed.run; the path has no
exchange step, so the ranks are independent replicas (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

# the oracle's BLAS may use every host core for the CPU baseline
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_frozen_projection_gb300 import workloads as wl  # noqa: E402

METRIC = "NVFP4 LoRA-linear fwd+dgrad TFLOPS (% FP4 peak); quant GB/s; layer tokens/s"
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor ratio on GB300
L2_FLUSH_BYTES = 256 << 20  # written between flushed repetitions (L2 is 129 MB)
# (N, K) of each distinct frozen-projection GEMM of the layer-3b step (out = M x N)
GEMM_SHAPES = {"q.fwd": (3072, 3072), "k.fwd": (1024, 3072), "v.fwd": (1024, 3072),
               "o.fwd": (3072, 3072), "gate_up.fwd": (16384, 3072), "down.fwd": (3072, 8192),
               "down.dgrad": (8192, 3072), "gate_up.dgrad": (3072, 16384),
               "o.dgrad": (3072, 3072), "q.dgrad": (3072, 3072), "k.dgrad": (3072, 1024),
               "v.dgrad": (3072, 1024)}
PROJS = ("q", "k", "v", "o", "gate_up", "down")
# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# gate|up forward GEMM with the SiLU statistics at 8192 tokens, from a one-pass ncu
# capture of that launch (profile_case gemm-gate-up-stats --m 8192), and the SHA-256
# of the sources and build script that kernel was compiled from when it was taken.
# The roofline reports it only while those files are unchanged, else null.
GU_FWD_TRAFFIC = {
    "bytes": 45287168 + 217468160,
    "tokens": 8192,
    "sources": ("nvfp4_frozen_projection_gb300/csrc/gemm.cu",
                "nvfp4_frozen_projection_gb300/csrc/tcgen05.cuh",
                "nvfp4_frozen_projection_gb300/csrc/common.cuh",
                "nvfp4_frozen_projection_gb300/csrc/kernels.h",
                "nvfp4_frozen_projection_gb300/build.py"),
    "sha256": "992159fdd64dbaf786ba81e33f97074b780bf2470ec31dc4174ccbd7270cbad8",
}
INPUTS = ("x", "attn", "dy", "dq", "dk", "dv")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [s.strip() for s in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.remove(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()),
                "samples": len(rows), "reasons": reasons}


# --------------------------------------------------------------------- oracle leg
def oracle_stack_sample(d, packs, rows: int):
    """The oracle chain of the layer-3b step (the same call sequence as the GPU
    step) over the first `rows` tokens.  Returns the GEMM FLOPs of the sample."""
    from oracle import chain
    sub = dict(d)
    for k in INPUTS:
        sub[k] = d[k][:rows]
    chain.decoder_layer(sub, packs)
    return wl.gemm_flops_per_step(5, m=rows)


def oracle_packs(d):
    import oracle as orc
    return {k: orc.pack_weight(d[k].W) for k in PROJS}


def cpu_baseline(d, rows=128, target_s=10.0):
    """Time the oracle (as it stands) on a bounded sample of the step."""
    packs = oracle_packs(d)
    oracle_stack_sample(d, packs, 16)  # warm caches / lazy loads
    n, t = 0, 0.0
    flops = 0.0
    t0 = time.perf_counter()
    while t < target_s or n == 0:
        flops += oracle_stack_sample(d, packs, rows)
        n += 1
        t = time.perf_counter() - t0
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"first {rows} tokens of the layer-3b step (fwd+dgrad chain, 12 FP64 "
                      f"GEMMs on exactly dequantised operands), {n} pass(es) in {t:.1f} s; "
                      "weight packs excluded (offline, as on the GPU)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    d = wl.layer3b()
    packs = oracle_packs(d)
    rows = 64
    for _ in range(args.warmup):
        oracle_stack_sample(d, packs, rows)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += oracle_stack_sample(d, packs, rows)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        # the launch's GPU count (the oracle itself runs on the host cores, rank 0 only)
        "n_gpus": int(os.environ.get("WORLD_SIZE", str(args.gpus))), "steps": args.steps,
        "warmup": args.warmup, "device": "host cores",
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(int(os.environ.get("WORLD_SIZE", str(args.gpus)))),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"each step: the first {rows} tokens of the layer-3b step "
                                   "(fwd+dgrad chain, FP64 GEMMs on exactly dequantised "
                                   "operands); TFLOP/s of that sample"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------- GPU leg
def build_stack(d, dev):
    import nvfp4_frozen_projection_gb300 as pk
    from nvfp4_frozen_projection_gb300.stack import DecoderProjectionStack

    stack = DecoderProjectionStack.from_workload(d, dev)
    torch.cuda.synchronize()
    pk.pact_check_status()
    return stack


def time_gemm_kernels(stack, inputs, reps):
    """Per-GEMM kernel time (CUDA events around the GEMM kernel alone, on the launch
    stream), the median over reps eager calls."""
    import nvfp4_frozen_projection_gb300 as pk
    x, attn, dy, dq, dk, dv = inputs
    stack.forward(x, attn)
    stack.backward(dy, dq, dk, dv)
    calls = {
        "q.fwd": lambda: stack.p["q"].forward(stack.xq1, stack.q),
        "k.fwd": lambda: stack.p["k"].forward(stack.xq1, stack.k),
        "v.fwd": lambda: stack.p["v"].forward(stack.xq1, stack.v),
        "o.fwd": lambda: stack.p["o"].forward(stack.attnq, stack.h1, residual=x),
        "gate_up.fwd": lambda: stack.p["gate_up"].forward_gate_up(stack.xq2, stack.gu,
                                                                  stack.gu_amax3),
        "down.fwd": lambda: stack.p["down"].forward(stack.hq, stack.out, residual=stack.h1),
        "down.dgrad": lambda: stack.p["down"].dgrad(stack.dyq, dy, stack.dh),
        "gate_up.dgrad": lambda: stack.p["gate_up"].dgrad(stack.dguq, stack.dgu, stack.dxn2),
        "o.dgrad": lambda: stack.p["o"].dgrad(stack.dh1q, stack.dh1, stack.dattn),
        "q.dgrad": lambda: stack.p["q"].dgrad(stack.dqq, dq, stack.dxn1),
        "k.dgrad": lambda: stack.p["k"].dgrad(stack.dkq, dk, stack.dxn1, accumulate=True),
        "v.dgrad": lambda: stack.p["v"].dgrad(stack.dvq, dv, stack.dxn1, accumulate=True),
    }
    m = stack.m
    flops = GEMM_SHAPES
    out = {}
    for name, fn in calls.items():
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for b, e in evs:  # torch creates the CUDA events on first record
            b.record()
            e.record()
        fn()
        torch.cuda.synchronize()
        _gpu_head_start()
        for b, e in evs:
            pk.pact_profile_next_gemm(b, e)
            fn()
        torch.cuda.synchronize()
        ms = statistics.median(b.elapsed_time(e) for b, e in evs)
        n_, k_ = flops[name]
        f = 2.0 * m * n_ * k_
        out[name] = {"ms": ms, "tflops": f / (ms * 1e-3) / 1e12, "flops": f}
    return out


def time_adapter_grads(stack, inputs, reps):
    """pact_lora_adapter_grad for each projection of the layer step, on the tensors a
    training step retains (CUDA events around each call)."""
    x, attn, dy, dq, dk, dv = inputs
    stack.forward(x, attn)
    stack.backward(dy, dq, dk, dv)
    p, m = stack.p, stack.m
    pairs = {"q": (stack.xq1, dq), "k": (stack.xq1, dk), "v": (stack.xq1, dv),
             "o": (stack.attnq, stack.dh1),
             "gate_up": (stack.xq2, stack.dgu), "down": (stack.hq, dy)}
    out, total = {}, 0.0
    for name, (xq, g) in pairs.items():
        proj = p[name]
        dA = torch.empty(proj.d_in, proj.A.shape[1], device=g.device, dtype=torch.float32)
        dB = torch.empty(proj.A.shape[1], proj.d_out, device=g.device, dtype=torch.float32)
        ms = time_call(lambda: proj.adapter_grad(xq, g, dA=dA, dB=dB), reps)
        one_pass = m * proj.d_in * (0.5 + 1 / 16) + m * proj.d_out * 2
        out[name] = {"ms": round(ms, 5), "one_pass_gbs": round(one_pass / (ms * 1e-3) / 1e9, 1)}
        total += ms
    out["total_ms"] = round(total, 5)
    return out


def time_bf16_comparator(m, shapes, reps):
    """The same GEMM shapes as plain BF16 matmuls through torch (cuBLAS): the BF16
    column of the pages' Table 1, for context.  shapes: name -> (N, K)."""
    out = {}
    for name, (n_, k_) in shapes.items():
        a = torch.randn(m, k_, device="cuda", dtype=torch.bfloat16)
        w = torch.randn(n_, k_, device="cuda", dtype=torch.bfloat16)
        y = torch.empty(m, n_, device="cuda", dtype=torch.bfloat16)
        for _ in range(3):
            torch.matmul(a, w.t(), out=y)
        torch.cuda.synchronize()
        b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b.record()
        for _ in range(reps):
            torch.matmul(a, w.t(), out=y)
        e.record()
        torch.cuda.synchronize()
        ms = b.elapsed_time(e) / reps
        out[name] = {"ms": ms, "tflops": 2.0 * m * n_ * k_ / (ms * 1e-3) / 1e12}
        del a, w, y
    torch.cuda.empty_cache()
    return out


def graph_of(fn):
    """fn captured in a CUDA graph (after one eager run that sizes its buffers)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


_FLUSH = None


def l2_flush():
    """Write a buffer twice the size of L2, evicting whatever it held."""
    global _FLUSH
    if _FLUSH is None:
        _FLUSH = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    _FLUSH.zero_()


def time_replays(run, reps, flush=False):
    """Median over reps runs of run(), each bracketed by CUDA events on the current
    stream; with flush, L2 is flushed before each run, outside the events."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    run()
    if flush:
        l2_flush()
    torch.cuda.synchronize()
    _gpu_head_start()
    for b, e in evs:
        if flush:
            l2_flush()
        b.record()
        run()
        e.record()
    torch.cuda.synchronize()
    return statistics.median(b.elapsed_time(e) for b, e in evs)


def _t32(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)


def _lin(p, dev, gate_up=False):
    from nvfp4_frozen_projection_gb300.stack import LoraLinear
    return LoraLinear(_t32(p.W, dev), _t32(p.A, dev).bfloat16(), _t32(p.B, dev).bfloat16(),
                      p.scale, gate_up=gate_up)


def _pass_line(name, tokens, gemm_flops, run, reps, extra=None):
    """One workload pass captured in a graph: median time warm and L2-flushed, GEMM
    TFLOP/s and tokens/s from the warm median."""
    g = graph_of(run)
    ms = time_replays(g.replay, reps)
    msf = time_replays(g.replay, reps, flush=True)
    line = {"tokens": tokens, "ms_median": round(ms, 5), "ms_median_l2_flushed": round(msf, 5),
            "gemm_tflops": round(gemm_flops / (ms * 1e-3) / 1e12, 1),
            "gemm_tflops_l2_flushed": round(gemm_flops / (msf * 1e-3) / 1e12, 1),
            "tokens_per_s": round(tokens / (ms * 1e-3), 1)}
    line.update(extra or {})
    del g
    return line


def config_lines(dev, reps):
    """Fwd + input-gradient passes of the other workloads, each its own sub-line:
    q-3b (one LoRA linear: X and dY quantised, forward, input gradient), mlp-3b
    (gate|up, SiLU-multiply, down and their input gradients), attn-1b (RMSNorm ->
    q/k/v forwards, their three input gradients accumulated, RMSNorm backward)."""
    import nvfp4_frozen_projection_gb300 as pk
    from nvfp4_frozen_projection_gb300 import NVFP4
    bf = dict(dtype=torch.bfloat16, device=dev)
    out = {}
    # q-3b
    d = wl.q3b()
    lin = _lin(d["proj"], dev)
    m, k = d["x"].shape
    x, dy = _t32(d["x"], dev).bfloat16(), _t32(d["dy"], dev).bfloat16()
    xq, dyq = NVFP4.empty(m, k, dev), NVFP4.empty(m, lin.d_out, dev)
    y, dx = torch.empty(m, lin.d_out, **bf), torch.empty(m, k, **bf)

    def q_pass():
        pk.pact_quant_nvfp4(x, out=xq)
        lin.forward(xq, y)
        lin.dgrad_q(dy, dyq, dx)
    out["q-3b"] = _pass_line("q-3b", m, 2 * lin.gemm_flops(m), q_pass, reps)
    del lin, x, dy, xq, dyq, y, dx
    # mlp-3b
    d = wl.mlp3b()
    gu_l, dn_l = _lin(d["gate_up"], dev, gate_up=True), _lin(d["down"], dev)
    m, h = d["x"].shape
    inter = dn_l.d_in
    x, dy = _t32(d["x"], dev).bfloat16(), _t32(d["dy"], dev).bfloat16()
    xq = NVFP4.empty(m, h, dev)
    gu = torch.empty(m, 2 * inter, **bf)
    hq, gq, uq = (NVFP4.empty(m, inter, dev) for _ in range(3))
    y = torch.empty(m, h, **bf)
    dyq, dh = NVFP4.empty(m, h, dev), torch.empty(m, inter, **bf)
    dgu, dguq = torch.empty(m, 2 * inter, **bf), NVFP4.empty(m, 2 * inter, dev)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    amax3 = torch.empty(3, dtype=torch.float32, device=dev)
    dx = torch.empty(m, h, **bf)

    def mlp_pass():
        pk.pact_quant_nvfp4(x, out=xq)
        gu_l.forward_gate_up(xq, gu, amax3)
        pk.pact_silu_mul_quant(gu, amax3=amax3, outs=(hq, gq, uq))
        dn_l.forward(hq, y)
        dn_l.dgrad_q(dy, dyq, dh)
        pk.pact_silu_mul_bwd(gq, uq, dh, dgateup=dgu, out_amax=amax)
        gu_l.dgrad_q(dgu, dguq, dx, amax=amax)
    out["mlp-3b"] = _pass_line("mlp-3b", m, 2 * (gu_l.gemm_flops(m) + dn_l.gemm_flops(m)),
                               mlp_pass, reps)
    del gu_l, dn_l, x, dy, xq, gu, hq, gq, uq, y, dyq, dh, dgu, dguq, dx
    # attn-1b
    d = wl.attn1b()
    lins = [_lin(p, dev) for p in d["projs"]]
    m, h = d["x"].shape
    x = _t32(d["x"], dev).bfloat16()
    gamma = _t32(d["gamma"], dev).bfloat16()
    dys = [_t32(a, dev).bfloat16() for a in d["dys"]]
    xq, rstd = NVFP4.empty(m, h, dev), torch.empty(m, dtype=torch.float32, device=dev)
    ys = [torch.empty(m, l.d_out, **bf) for l in lins]
    dyqs = [NVFP4.empty(m, l.d_out, dev) for l in lins]
    dn, dxx = torch.empty(m, h, **bf), torch.empty(m, h, **bf)
    eps = float(d["eps"])

    def attn_pass():
        pk.pact_rmsnorm_quant(x, gamma, eps, out=xq, rstd=rstd)
        for l, yy in zip(lins, ys):
            l.forward(xq, yy)
        for i, (l, dy_, dyq_) in enumerate(zip(lins, dys, dyqs)):
            l.dgrad_q(dy_, dyq_, dn, accumulate=i > 0)
        pk.pact_rmsnorm_bwd(xq, gamma, rstd, dn, dx=dxx)
    out["attn-1b"] = _pass_line("attn-1b", m, 2 * sum(l.gemm_flops(m) for l in lins), attn_pass,
                                reps)
    del lins, x, dys, xq, ys, dyqs, dn, dxx
    torch.cuda.empty_cache()
    return out


def layer_1b_projection(dev, reps, m=26 * 1024):
    """The decoder-layer projection stack at Llama-1B shapes (hidden 2048, 32 q heads
    / 8 kv heads of 64, intermediate 8192, r = 16), batch 26 x 1024, with weights and
    inputs drawn on the device (normal draws of the workload scales; the values do not
    change the work).  Returns the step's median time."""
    from nvfp4_frozen_projection_gb300.stack import DecoderProjectionStack, LoraLinear
    gen = torch.Generator(device=dev)
    gen.manual_seed(1016)
    hid, kv, inter, r = 2048, 512, 8192, 16

    def lin(d_in, d_out, rr=r, gate_up=False):
        W = torch.randn(d_out, d_in, device=dev, generator=gen) * 0.02
        A = (torch.randn(d_in, rr, device=dev, generator=gen) / d_in ** 0.5).bfloat16()
        B = (torch.randn(rr, d_out, device=dev, generator=gen) * 0.1).bfloat16()
        return LoraLinear(W, A, B, 2.0, gate_up=gate_up)
    proj = {"q": lin(hid, hid), "k": lin(hid, kv), "v": lin(hid, kv), "o": lin(hid, hid),
            "gate_up": lin(hid, 2 * inter, 2 * r, gate_up=True), "down": lin(inter, hid)}
    g1 = (1 + 0.1 * torch.randn(hid, device=dev, generator=gen)).bfloat16()
    g2 = (1 + 0.1 * torch.randn(hid, device=dev, generator=gen)).bfloat16()
    st = DecoderProjectionStack(m, proj, g1, g2, 1e-5)
    x = torch.randn(m, hid, device=dev, generator=gen).bfloat16()
    attn = torch.randn(m, hid, device=dev, generator=gen).bfloat16()
    dy, dq = ((torch.randn(m, hid, device=dev, generator=gen) * 0.01).bfloat16() for _ in range(2))
    dk, dv = ((torch.randn(m, kv, device=dev, generator=gen) * 0.01).bfloat16() for _ in range(2))

    def step():
        st.forward(x, attn)
        st.backward(dy, dq, dk, dv)
    g = graph_of(step)
    ms = time_replays(g.replay, reps)
    flops = st.gemm_flops()
    del g, st, proj
    torch.cuda.empty_cache()
    return ms, flops


def _gpu_head_start():
    """Keep the GPU busy for a few ms so the host enqueues every rep before the GPU
    reaches it: the events then time GPU execution, not host launch latency."""
    torch.cuda._sleep(20_000_000)


def time_call(fn, reps):
    """Median of reps eager calls (CUDA events around each)."""
    return time_replays(fn, reps)


# ------------------------------------------------------------------ multi-rank
def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time: every rank runs an independent replica of the step
    (no data-path collective), so the job takes as long as its slowest rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Units processed by all ranks per second (weak scaling: each rank does the
    same fixed amount of work)."""
    return units_per_rank * world / (ms * 1e-3)


def step_config(world: int) -> dict:
    """The workload's configuration, the same on both arms: the layer-3b step at 8192
    tokens, whatever sample of it an arm times."""
    return {"workload": "layer-3b", "tokens_per_step": 8192, "hidden": 3072,
            "intermediate": 8192, "q_kv_o": [3072, 1024, 1024, 3072], "r": 16,
            "gemms_per_step": 12, "fused": "gate|up runs as one GEMM",
            "gemm_flops_per_step": wl.gemm_flops_per_step(5, m=8192),
            "l2": "no flush between timed steps: one step moves several GB through HBM "
                  "(L2 is 129 MB); ms_per_step_l2_flushed flushes before every step",
            "parallelism": f"replicas x{world}"}


def sources_sha256(paths) -> str:
    """SHA-256 over the given repository files, in order."""
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def dominant_traffic(dominant: str, tokens: int):
    """Per-launch DRAM bytes of the dominant GEMM from the stored capture, or None
    when the capture does not cover this kernel, size or build."""
    t = GU_FWD_TRAFFIC
    if dominant != "gate_up.fwd" or tokens != t["tokens"]:
        return None
    return t["bytes"] if sources_sha256(t["sources"]) == t["sha256"] else None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-graph", action="store_true", help="replay the step eagerly")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from nvfp4_frozen_projection_gb300 import build as pkbuild
    pkbuild.build()
    import nvfp4_frozen_projection_gb300 as pk
    if not pk.pact_device_supported():
        raise RuntimeError(pk.load_library().pact_last_error().decode())

    d = wl.layer3b()
    stack = build_stack(d, dev)
    host_in = [torch.from_numpy(np.ascontiguousarray(d[n], np.float32)).bfloat16().pin_memory()
               for n in INPUTS]
    inputs = [h.to(dev) for h in host_in]
    x, attn, dy, dq, dk, dv = inputs

    def step():
        stack.forward(x, attn)
        stack.backward(dy, dq, dk, dv)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    pk.pact_check_status()

    graph = None
    n0 = pk.pact_launch_count()
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        launches_per_step = pk.pact_launch_count() - n0
        # the two replays before the timed region are what a profiler started with
        # collection off (ncu --profile-from-start off) records
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        run = graph.replay
    else:
        step()
        launches_per_step = pk.pact_launch_count() - n0
        run = step

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---------------- timed region: K steps, inputs resident in HBM.  The clock
    # sampler runs through a one-second soak of the same replays just before the
    # timed region and through the region itself, so it sees the GPU under this load
    # however short K steps are.  Each step is also bracketed by its own events for
    # the per-step median.
    barrier()
    torch.cuda.synchronize()
    step_evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 1.0:
            for _ in range(20):
                run()
            torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_begin.record()
        for i in range(args.steps):
            step_evs[i].record()
            run()
        step_evs[args.steps].record()
        t_end.record()
        torch.cuda.synchronize()
    barrier()
    ms = t_begin.elapsed_time(t_end) / args.steps
    ms_median = statistics.median(step_evs[i].elapsed_time(step_evs[i + 1])
                                  for i in range(args.steps))
    clocks = clk.summary()
    clocks["window"] = "1 s of the same step replays just before the timed region, then the region"
    # the same step with L2 flushed before each replay (outside its events)
    ms_flushed = time_replays(run, max(10, min(args.steps, 50)), flush=True)
    pk.pact_check_status()
    ms = max_over_ranks(ms, dev)

    flops = stack.gemm_flops()
    value = job_throughput(flops, world, ms) / 1e12
    tokens_per_s = job_throughput(stack.m, world, ms)

    # ---------------- end to end: pinned host inputs in, result (dx) out, every step.
    # As a training loop would run it: two sets of device buffers (a second stack
    # sharing the packed weights, each with its own captured step), the next step's
    # inputs uploaded on one copy stream while this step computes, and each step's
    # result read back on another while the next one computes.
    from nvfp4_frozen_projection_gb300.stack import DecoderProjectionStack
    stack2 = DecoderProjectionStack(stack.m, stack.p, stack.gamma1, stack.gamma2, stack.eps)
    inputs2 = [torch.empty_like(t) for t in inputs]
    sets = [(stack, inputs), (stack2, inputs2)]
    runs = []
    for st, ins in sets:
        def step_on(st=st, ins=ins):
            st.forward(ins[0], ins[1])
            st.backward(*ins[2:])
        if graph is not None and st is stack:
            runs.append(run)
            continue
        for t_dev, h in zip(ins, host_in):
            t_dev.copy_(h)
        step_on()
        torch.cuda.synchronize()
        if graph is not None:
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2):
                step_on()
            runs.append(g2.replay)
        else:
            runs.append(step_on)
    host_out = [torch.empty_like(stack.dx, device="cpu").pin_memory() for _ in range(2)]
    compute = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def upload(b, after=None):
        with torch.cuda.stream(up):
            if after is not None:
                up.wait_event(after)  # the step that last read buffer b has finished
            for h, t_dev in zip(host_in, sets[b][1]):
                t_dev.copy_(h, non_blocking=True)
            ev_in[b].record(up)

    barrier()
    torch.cuda.synchronize()
    e_begin, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_begin.record(compute)
    up.wait_stream(compute)
    down.wait_stream(compute)
    upload(0)
    for i in range(args.steps):
        b = i % 2
        if i + 1 < args.steps:
            upload(1 - b, ev_done[1 - b] if i >= 1 else None)
        compute.wait_event(ev_in[b])
        if i >= 2:
            compute.wait_event(ev_out[b])  # step i-2's result has left this buffer
        runs[b]()
        ev_done[b].record(compute)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[b])
            host_out[b].copy_(sets[b][0].dx, non_blocking=True)
            ev_out[b].record(down)
    compute.wait_stream(up)
    compute.wait_stream(down)
    e_end.record(compute)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = max_over_ranks(e_begin.elapsed_time(e_end) / args.steps, dev)
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()

    # ---------------- per-kernel live timing (GEMM kernels alone; quantiser)
    kern = time_gemm_kernels(stack, inputs, reps=max(5, args.steps // 2))
    P, src = peaks()
    fp4_peak = P["bf16_tflops"] * FP4_OVER_BF16
    step_share = {k: v["ms"] for k, v in kern.items()}
    dominant = max(step_share, key=step_share.get)
    dk_ = kern[dominant]
    m, hid = stack.m, stack.hidden
    cfg = step_config(world)
    assert cfg["tokens_per_step"] == m and cfg["gemm_flops_per_step"] == flops, \
        "the stack and the reported configuration disagree"
    # memory-bound calls alone: algorithmic bytes (inputs read once, outputs written
    # once) over the median call time, warm and with L2 flushed before each call
    mem_calls = {
        "quant_nvfp4 8192x3072": (lambda: pk.pact_quant_nvfp4(dy, out=stack.dyq),
                                  m * hid * (2 + 0.5 + 1 / 16)),
        "rmsnorm_quant 8192x3072": (lambda: pk.pact_rmsnorm_quant(
            x, stack.gamma1, stack.eps, out=stack.xq1, rstd=stack.rstd1),
            m * hid * (2 + 0.5 + 1 / 16) + 4 * m),
        "silu_mul_quant 8192x2x8192": (lambda: pk.pact_silu_mul_quant(
            stack.gu, outs=(stack.hq, stack.gq, stack.uq)), m * stack.inter * (4 + 3 * (0.5 + 1 / 16))),
        # as the step runs it: the gate|up GEMM's epilogue supplied the amaxes
        "silu_mul_quant 8192x2x8192 (amax from the GEMM)": (lambda: pk.pact_silu_mul_quant(
            stack.gu, amax3=stack.gu_amax3, outs=(stack.hq, stack.gq, stack.uq)),
            m * stack.inter * (4 + 3 * (0.5 + 1 / 16))),
        "silu_mul_bwd 8192x8192": (lambda: pk.pact_silu_mul_bwd(
            stack.gq, stack.uq, stack.dh, dgateup=stack.dgu, out_amax=stack.dgu_amax),
            m * stack.inter * (2 * (0.5 + 1 / 16) + 2 + 4)),
        "rmsnorm_bwd 8192x3072 (+dres)": (lambda: pk.pact_rmsnorm_bwd(
            stack.xq2, stack.gamma2, stack.rstd2, stack.dxn2, dres=dy, dx=stack.dh1,
            out_amax=stack.dh1_amax), m * hid * ((0.5 + 1 / 16) + 2 + 2 + 2) + 4 * m),
    }
    memory_kernels = {}
    for name, (fn, nbytes) in mem_calls.items():
        a = time_replays(fn, 20)
        b = time_replays(fn, 20, flush=True)
        memory_kernels[name] = {"ms": round(a, 5), "gbs": round(nbytes / (a * 1e-3) / 1e9, 1),
                                "ms_l2_flushed": round(b, 5),
                                "gbs_l2_flushed": round(nbytes / (b * 1e-3) / 1e9, 1)}
    memory_kernels["hbm_peak_gbs"] = P["hbm_gbs"]
    q_ms, q_bytes = memory_kernels["quant_nvfp4 8192x3072"]["ms"], mem_calls["quant_nvfp4 8192x3072"][1]
    pk.pact_check_status()
    adapter = time_adapter_grads(stack, inputs, reps=10)
    bf16 = time_bf16_comparator(m, GEMM_SHAPES, reps=10)
    configs = config_lines(dev, reps=20)
    ms_1b, flops_1b = layer_1b_projection(dev, reps=10)
    pk.pact_check_status()

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4", "data": "synthetic",
        "config": cfg,
        "graph": graph is not None,
        "ms_per_step_median": ms_median,
        "ms_per_step_l2_flushed": ms_flushed,
        "clocks": clocks,
        "e2e": {"value": job_throughput(flops, world, ms_e2e) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e},
        "gpu_launches": int(launches_per_step) * args.steps,
        "layer_tokens_per_s": tokens_per_s,
        "fp4_peak_frac_step": value / world / fp4_peak,
        "roofline": {"bound": "tensor", "kernel": f"k_gemm_nvfp4 ({dominant})",
                     "achieved": dk_["tflops"], "peak": fp4_peak, "unit": "TFLOP/s",
                     "frac": dk_["tflops"] / fp4_peak,
                     "traffic": dominant_traffic(dominant, m),
                     "peak_source": f"{src} bf16 burst x {FP4_OVER_BF16:g} (nominal FP4:BF16)"},
        "gemm_kernels": {k: {"ms": round(v["ms"], 5), "tflops": round(v["tflops"], 1)}
                         for k, v in kern.items()},
        "memory_kernels": memory_kernels,
        # the other workloads' fwd + input-gradient passes (graph replays; medians)
        "configs": configs,
        # model tokens/s projected from one layer's projection stack (attention core,
        # embeddings, LM head and optimizer excluded): layer-3b x 28 layers, and a
        # Llama-1B-shaped stack at 26 x 1024 tokens x 16 layers
        "projected_model_tokens_per_s": {
            "llama-3b (28 layers, layer-3b step)": round(m / (28 * ms_median * 1e-3), 1),
            "llama-1b (16 layers, 1B-shaped stack, 26624 tokens)": round(
                26 * 1024 / (16 * ms_1b * 1e-3), 1),
            "layer-1b step ms": round(ms_1b, 5),
            "layer-1b gemm_tflops": round(flops_1b / (ms_1b * 1e-3) / 1e12, 1)},
        "quant_gbs": q_bytes / (q_ms * 1e-3) / 1e9,
        # the LoRA adapter gradients dA, dB of the seven projections (outside the
        # fwd+dgrad step that the metric times): per call, and bandwidth against one
        # read of the NVFP4 input and of the BF16 output gradient
        "adapter_grad": adapter,
        # context: the same GEMM shapes as cuBLAS BF16 matmuls (no LoRA, no epilogue
        # work), and the NVFP4 kernel's speedup over them
        "bf16_comparator": {k: {"ms": round(v["ms"], 5), "tflops": round(v["tflops"], 1),
                                "nvfp4_speedup": round(v["ms"] / kern[k]["ms"], 2)}
                            for k, v in bf16.items()},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(d)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
