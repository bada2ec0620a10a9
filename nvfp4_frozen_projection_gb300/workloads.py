"""Seeded synthetic inputs for the five workloads of the NVFP4 LoRA linear.

This module only draws random numbers and rounds them to the storage type; it holds
none of the method's arithmetic, so it may feed both the CUDA library and the CPU
oracle.  Every array is drawn in FP32 with numpy's PCG64 generator (seed = 1000 +
workload index) and BF16 tensors are the round-to-nearest-even BF16 of that draw.
The paper's own workloads are fine-tuning datasets at sequence length 1024
(Table 5); these synthetic tensors stand in for them by shape and distribution.

Workloads (M = tokens):
  1 tiny      M=64, 256 -> 256, r=8, alpha=16
  2 q-3b      M=4096, 3072 -> 3072, r=16, alpha=32, X with 0.1% outlier channels x20
  3 mlp-3b    M=4096, gate|up 3072 -> 2x8192 (one fused GEMM), down 8192 -> 3072
  4 attn-1b   M=26624, RMSNorm(2048) -> q 2048, k 512, v 512
  5 layer-3b  M=8192, RMSNorm -> q/k/v 3072/1024/1024, o 3072, RMSNorm -> gate|up, down
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def bf16_round(a: np.ndarray) -> np.ndarray:
    """FP32 values rounded to the nearest BF16 (ties to even), returned as FP32."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def to_bf16_tensor(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def rng_for(index: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(1000 + index + 100 * salt))


def normal(rng, shape, std) -> np.ndarray:
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def student_t_unit_rms(rng, shape, nu=3.0) -> np.ndarray:
    """Student-t (nu) draws scaled by their empirical global rms to unit rms."""
    x = rng.standard_t(nu, size=shape).astype(np.float32)
    rms = np.float32(np.sqrt(np.mean(x.astype(np.float64) ** 2)))
    return (x / rms).astype(np.float32)


def with_outlier_channels(rng, x: np.ndarray, frac=0.001, factor=20.0) -> np.ndarray:
    """Scale round(frac * d_in) (at least 1) seeded channels of x by factor."""
    d = x.shape[1]
    n = max(1, int(round(frac * d)))
    ch = rng.choice(d, size=n, replace=False)
    x = x.copy()
    x[:, ch] *= np.float32(factor)
    return x


@dataclass
class Proj:
    """One LoRA linear: W [d_out, d_in] FP32 (frozen, RTN-quantised), A [d_in, r] and
    B [r, d_out] BF16 adapters; applied scale = alpha / r."""
    name: str
    d_in: int
    d_out: int
    r: int
    alpha: float
    W: np.ndarray = field(repr=False, default=None)
    A: np.ndarray = field(repr=False, default=None)
    B: np.ndarray = field(repr=False, default=None)

    @property
    def scale(self) -> float:
        return float(self.alpha) / float(self.r)


def make_proj(rng, name, d_in, d_out, r, alpha, w_std, b_std=0.1) -> Proj:
    p = Proj(name, d_in, d_out, r, alpha)
    p.W = normal(rng, (d_out, d_in), w_std)
    p.A = bf16_round(normal(rng, (d_in, r), 1.0 / np.sqrt(d_in)))
    p.B = bf16_round(normal(rng, (r, d_out), b_std))
    return p


def fuse_outputs(name: str, parts: list) -> Proj:
    """Projections of one input as one GEMM: W stacked along the outputs (one frozen
    weight, so one per-tensor scale), A side by side, B block-diagonal.  Each part's
    LoRA scale alpha/r is kept, so every output column gets exactly its own
    adapter's term."""
    r, alpha = parts[0].r, parts[0].alpha
    assert all(q.r == r and q.alpha == alpha and q.d_in == parts[0].d_in for q in parts)
    n = len(parts)
    p = Proj(name, parts[0].d_in, sum(q.d_out for q in parts), n * r, alpha * n)
    p.W = np.concatenate([q.W for q in parts], axis=0)
    p.A = np.concatenate([q.A for q in parts], axis=1)
    B = np.zeros((n * r, p.d_out), np.float32)
    c = 0
    for i, q in enumerate(parts):
        B[i * r:(i + 1) * r, c:c + q.d_out] = q.B
        c += q.d_out
    p.B = B
    return p


def fuse_gate_up(gate: Proj, up: Proj) -> Proj:
    """gate and up as one [2I, H] GEMM (see fuse_outputs)."""
    return fuse_outputs("gate_up", [gate, up])


WORKLOAD_NAMES = {1: "tiny", 2: "q-3b", 3: "mlp-3b", 4: "attn-1b", 5: "layer-3b"}


def tiny(m: int = 64):
    """Workload 1: single LoRA linear, M=64, 256 -> 256, r=8, alpha=16."""
    rng = rng_for(1)
    d = 256
    x = bf16_round(normal(rng, (m, d), 1.0))
    p = make_proj(rng, "proj", d, d, 8, 16.0, w_std=1.0 / np.sqrt(d))
    dy = bf16_round(normal(rng, (m, d), 1.0))
    return dict(x=x, proj=p, dy=dy)


def q3b(m: int = 4096):
    """Workload 2: Llama-3B query projection."""
    rng = rng_for(2)
    d = 3072
    x = with_outlier_channels(rng, normal(rng, (m, d), 1.0))
    x = bf16_round(x)
    p = make_proj(rng, "q", d, d, 16, 32.0, w_std=0.02)
    dy = bf16_round(normal(rng, (m, d), 1e-2))
    return dict(x=x, proj=p, dy=dy)


def mlp3b(m: int = 4096, hidden: int = 3072, inter: int = 8192):
    """Workload 3: Llama-3B MLP (gate|up fused, SiLU-multiply, down)."""
    rng = rng_for(3)
    x = bf16_round(normal(rng, (m, hidden), 1.0))
    gate = make_proj(rng, "gate", hidden, inter, 16, 32.0, w_std=0.02)
    up = make_proj(rng, "up", hidden, inter, 16, 32.0, w_std=0.02)
    down = make_proj(rng, "down", inter, hidden, 16, 32.0, w_std=0.02)
    dy = bf16_round(normal(rng, (m, hidden), 1e-2))
    return dict(x=x, gate_up=fuse_gate_up(gate, up), down=down, dy=dy)


def attn1b(m: int = 26624, hidden: int = 2048, kv: int = 512):
    """Workload 4: Llama-1B attention-input projections behind the fused RMSNorm."""
    rng = rng_for(4)
    x = bf16_round(student_t_unit_rms(rng, (m, hidden)))
    gamma = bf16_round(1.0 + normal(rng, (hidden,), 0.1))
    projs = [make_proj(rng, "q", hidden, hidden, 16, 32.0, w_std=0.02),
             make_proj(rng, "k", hidden, kv, 16, 32.0, w_std=0.02),
             make_proj(rng, "v", hidden, kv, 16, 32.0, w_std=0.02)]
    dys = [bf16_round(normal(rng, (m, p.d_out), 1e-2)) for p in projs]
    return dict(x=x, gamma=gamma, projs=projs, dys=dys, eps=np.float32(1e-5))


def layer3b(m: int = 8192, hidden: int = 3072, kv: int = 1024, inter: int = 8192):
    """Workload 5: Llama-3B decoder-layer projection stack.  The attention core is
    replaced by a seeded N(0,1) BF16 tensor; the gradients flowing into q/k/v from
    the (out of scope) attention backward are seeded N(0, 1e-2^2) tensors.  q, k
    and v are separate projections (each its own frozen weight and per-tensor
    scale, each incoming gradient its own tensor); gate and up run as the fused
    projection gate_up."""
    rng = rng_for(5)
    x = bf16_round(student_t_unit_rms(rng, (m, hidden)))
    gamma1 = bf16_round(1.0 + normal(rng, (hidden,), 0.1))
    gamma2 = bf16_round(1.0 + normal(rng, (hidden,), 0.1))
    q = make_proj(rng, "q", hidden, hidden, 16, 32.0, w_std=0.02)
    k = make_proj(rng, "k", hidden, kv, 16, 32.0, w_std=0.02)
    v = make_proj(rng, "v", hidden, kv, 16, 32.0, w_std=0.02)
    o = make_proj(rng, "o", hidden, hidden, 16, 32.0, w_std=0.02)
    gate = make_proj(rng, "gate", hidden, inter, 16, 32.0, w_std=0.02)
    up = make_proj(rng, "up", hidden, inter, 16, 32.0, w_std=0.02)
    down = make_proj(rng, "down", inter, hidden, 16, 32.0, w_std=0.02)
    attn = bf16_round(normal(rng, (m, hidden), 1.0))
    dy = bf16_round(normal(rng, (m, hidden), 1e-2))
    dq = bf16_round(normal(rng, (m, hidden), 1e-2))
    dk = bf16_round(normal(rng, (m, kv), 1e-2))
    dv = bf16_round(normal(rng, (m, kv), 1e-2))
    return dict(x=x, gamma1=gamma1, gamma2=gamma2, q=q, k=k, v=v, o=o,
                gate_up=fuse_gate_up(gate, up), down=down, attn=attn,
                dy=dy, dq=dq, dk=dk, dv=dv, eps=np.float32(1e-5))


def gemm_flops_per_step(which: int, m: int | None = None) -> float:
    """2*M*N*K summed over the frozen-projection GEMMs of one fwd+dgrad pass."""
    shapes = {
        1: (64, [(256, 256)]),
        2: (4096, [(3072, 3072)]),
        3: (4096, [(3072, 16384), (8192, 3072)]),
        4: (26624, [(2048, 2048), (2048, 512), (2048, 512)]),
        5: (8192, [(3072, 3072), (3072, 1024), (3072, 1024), (3072, 3072),
                   (3072, 16384), (8192, 3072)]),
    }[which]
    mm = shapes[0] if m is None else m
    return float(sum(2 * 2 * mm * k * n for (k, n) in shapes[1]))
