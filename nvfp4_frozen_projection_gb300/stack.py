"""LoRA linear layers and the decoder-layer projection stack built on libpact.

"PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs", Figure 2 (decoder data
flow) and Table 7 (precision allocation): RMSNorm -> NVFP4 feeds the q/k/v
projections, the attention output feeds o, a residual add, RMSNorm -> NVFP4 feeds
the fused gate/up projection, SiLU-multiply -> NVFP4 feeds down, and a second
residual add.  Attention and its backward are out of scope: the attention output
and the gradients flowing back into q/k/v are given tensors.

Every operation here is a libpact call; this module only owns buffers and the
order of calls.  Buffers are allocated once, so one step can be captured in a
CUDA graph and replayed.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (NVFP4, pact_lora_linear_dgrad, pact_lora_linear_dgrad_q, pact_lora_linear_fwd,
               pact_lora_linear_fwd_gate_up, pact_pack_weight_bwd, pact_pack_weight_fwd_gate_up,
               pact_lora_adapter_grad, pact_pack_weight_fwd, pact_quant_nvfp4, pact_rmsnorm_bwd,
               pact_rmsnorm_quant,
               pact_silu_mul_bwd, pact_silu_mul_quant)


class LoraLinear:
    """Frozen weight W [d_out, d_in] packed once into the cached forward and backward
    NVFP4 layouts, BF16 adapters A [d_in, r] and B [r, d_out], scale = alpha / r.
    gate_up: W is a fused [gate; up] weight whose forward also yields the SiLU
    statistics of its output (forward_gate_up)."""

    def __init__(self, W: torch.Tensor, A: torch.Tensor, B: torch.Tensor, scale: float,
                 gate_up: bool = False):
        self.d_out, self.d_in = W.shape
        self.gate_up = gate_up
        self.w_fwd = pact_pack_weight_fwd_gate_up(W) if gate_up else pact_pack_weight_fwd(W)
        self.w_bwd = pact_pack_weight_bwd(W)
        self.A, self.B, self.scale = A, B, float(scale)

    def forward(self, xq: NVFP4, y: torch.Tensor, residual=None, out_amax=None):
        if self.gate_up:
            raise ValueError("a gate|up projection runs forward_gate_up")
        return pact_lora_linear_fwd(xq, self.w_fwd, self.A, self.B, self.scale,
                                    residual=residual, y=y, out_amax=out_amax)

    def forward_gate_up(self, xq: NVFP4, y: torch.Tensor, amax3: torch.Tensor):
        """y = [gate | up], amax3 = (max |silu(gate) up|, max |gate|, max |up|)."""
        return pact_lora_linear_fwd_gate_up(xq, self.w_fwd, self.A, self.B, self.scale, y=y,
                                            amax3=amax3)

    def dgrad(self, dyq: NVFP4, dy: torch.Tensor, dx: torch.Tensor, accumulate=False):
        return pact_lora_linear_dgrad(dyq, dy, self.w_bwd, self.A, self.B, self.scale, dx=dx,
                                      accumulate=accumulate)

    def dgrad_q(self, dy: torch.Tensor, dyq: NVFP4, dx: torch.Tensor, amax=None,
                accumulate=False):
        """Quantise dy into dyq and run the input gradient, in one pass over dy."""
        return pact_lora_linear_dgrad_q(dy, self.w_bwd, self.A, self.B, self.scale, amax=amax,
                                        dyq=dyq, dx=dx, accumulate=accumulate)

    def adapter_grad(self, xq: NVFP4, dy: torch.Tensor, dA=None, dB=None):
        return pact_lora_adapter_grad(xq, dy, self.A, self.B, self.scale, dA=dA, dB=dB)

    def gemm_flops(self, m: int) -> float:
        return 2.0 * m * self.d_in * self.d_out


class DecoderProjectionStack:
    """The seven LoRA projections of a Llama decoder layer with both RMSNorms, the
    SiLU-multiply and the two residual adds; forward and input-gradient pass.
    q, k and v are separate projections, each with its own frozen weight and
    per-tensor scales; gate and up run as one fused GEMM (gate_up), adapters side
    by side and B block-diagonal."""

    def __init__(self, m: int, proj: dict, gamma1, gamma2, eps: float = 1e-5,
                 concurrent: bool = True):
        self.m = m
        self.concurrent = concurrent
        self._side_streams = []
        self.p = proj  # q, k, v, o, gate_up, down -> LoraLinear
        self.gamma1, self.gamma2, self.eps = gamma1, gamma2, float(eps)
        hidden = proj["q"].d_in
        inter = proj["down"].d_in
        dev = gamma1.device
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.hidden, self.inter = hidden, inter
        # forward state (the NVFP4 tensors are what backward reuses)
        self.xq1 = NVFP4.empty(m, hidden, dev)
        self.rstd1 = torch.empty(m, dtype=torch.float32, device=dev)
        self.q = torch.empty(m, proj["q"].d_out, **bf)
        self.k = torch.empty(m, proj["k"].d_out, **bf)
        self.v = torch.empty(m, proj["v"].d_out, **bf)
        self.attnq = NVFP4.empty(m, hidden, dev)
        self.h1 = torch.empty(m, hidden, **bf)
        self.xq2 = NVFP4.empty(m, hidden, dev)
        self.rstd2 = torch.empty(m, dtype=torch.float32, device=dev)
        self.gu = torch.empty(m, 2 * inter, **bf)
        self.gu_amax3 = torch.empty(3, dtype=torch.float32, device=dev)
        self.hq = NVFP4.empty(m, inter, dev)
        self.gq = NVFP4.empty(m, inter, dev)
        self.uq = NVFP4.empty(m, inter, dev)
        self.out = torch.empty(m, hidden, **bf)
        # backward state
        self.dyq = NVFP4.empty(m, hidden, dev)
        self.dh = torch.empty(m, inter, **bf)
        self.dgu = torch.empty(m, 2 * inter, **bf)
        self.dgu_amax = torch.empty(1, dtype=torch.float32, device=dev)
        self.dh1_amax = torch.empty(1, dtype=torch.float32, device=dev)
        self.dguq = NVFP4.empty(m, 2 * inter, dev)
        self.dxn2 = torch.empty(m, hidden, **bf)
        self.dh1 = torch.empty(m, hidden, **bf)
        self.dh1q = NVFP4.empty(m, hidden, dev)
        self.dattn = torch.empty(m, hidden, **bf)
        self.dqq = NVFP4.empty(m, proj["q"].d_out, dev)
        self.dkq = NVFP4.empty(m, proj["k"].d_out, dev)
        self.dvq = NVFP4.empty(m, proj["v"].d_out, dev)
        self.dxn1 = torch.empty(m, hidden, **bf)
        self.dx = torch.empty(m, hidden, **bf)

    def _side(self, i: int = 0):
        """Side stream i for work independent of the main chain: its kernels fill
        the SMs that a persistent GEMM's last tiles leave idle.  Forked from and
        joined back into the current stream, so graph capture records every branch."""
        if self.concurrent is False:
            return None
        while len(self._side_streams) <= i:
            self._side_streams.append(torch.cuda.Stream(device=self.gamma1.device))
        return self._side_streams[i]

    def forward(self, x: torch.Tensor, attn: torch.Tensor) -> torch.Tensor:
        p = self.p
        main, side = torch.cuda.current_stream(), self._side()
        if side is not None:
            side.wait_stream(main)
            with torch.cuda.stream(side):
                # attention core (out of scope): its output is the given tensor attn
                pact_quant_nvfp4(attn, out=self.attnq)
                p["o"].forward(self.attnq, self.h1, residual=x)
        pact_rmsnorm_quant(x, self.gamma1, self.eps, out=self.xq1, rstd=self.rstd1)
        side2 = self._side(1)
        if side2 is not None:  # q, k and v all read xq1 only: run them side by side
            side2.wait_stream(main)
            with torch.cuda.stream(side2):
                p["k"].forward(self.xq1, self.k)
                p["v"].forward(self.xq1, self.v)
        p["q"].forward(self.xq1, self.q)
        if side2 is None:
            p["k"].forward(self.xq1, self.k)
            p["v"].forward(self.xq1, self.v)
        else:
            main.wait_stream(side2)
        if side is None:
            pact_quant_nvfp4(attn, out=self.attnq)
            p["o"].forward(self.attnq, self.h1, residual=x)
        else:
            main.wait_stream(side)
        pact_rmsnorm_quant(self.h1, self.gamma2, self.eps, out=self.xq2, rstd=self.rstd2)
        # the gate|up GEMM's epilogue yields the three amaxes: one pass of SiLU-multiply
        p["gate_up"].forward_gate_up(self.xq2, self.gu, self.gu_amax3)
        pact_silu_mul_quant(self.gu, amax3=self.gu_amax3, outs=(self.hq, self.gq, self.uq))
        p["down"].forward(self.hq, self.out, residual=self.h1)
        return self.out

    def adapter_grads(self, dy, dq, dk, dv) -> dict:
        """dA, dB of all seven adapters from the tensors the forward and backward
        retained (call after backward): each projection's NVFP4 input and the BF16
        gradient of its output.  For the fused projections the adapters' gradients
        are the diagonal blocks of dB (and the matching columns of dA)."""
        p = self.p
        pairs = {"q": (self.xq1, dq), "k": (self.xq1, dk), "v": (self.xq1, dv),
                 "o": (self.attnq, self.dh1),
                 "gate_up": (self.xq2, self.dgu), "down": (self.hq, dy)}
        return {name: p[name].adapter_grad(xq, g) for name, (xq, g) in pairs.items()}

    def backward(self, dy, dq, dk, dv) -> torch.Tensor:
        """dy: gradient of the layer output; dq, dk, dv: the gradients flowing back
        from the (out of scope) attention core into the q, k, v outputs."""
        p = self.p
        main, side = torch.cuda.current_stream(), self._side()
        # every input gradient quantises its dY in the same pass that forms the
        # LoRA down-projection (pact_lora_linear_dgrad_q).  The q, k and v input
        # gradients need only the attention core's gradients: they run beside the
        # down -> SiLU -> gate|up -> RMSNorm -> o chain, accumulating into one
        # buffer in the order q, k, v.
        if side is not None:
            side.wait_stream(main)
            with torch.cuda.stream(side):
                self._qkv_dgrad(dq, dk, dv)
        p["down"].dgrad_q(dy, self.dyq, self.dh)
        pact_silu_mul_bwd(self.gq, self.uq, self.dh, dgateup=self.dgu, out_amax=self.dgu_amax)
        p["gate_up"].dgrad_q(self.dgu, self.dguq, self.dxn2, amax=self.dgu_amax)
        pact_rmsnorm_bwd(self.xq2, self.gamma2, self.rstd2, self.dxn2, dres=dy, dx=self.dh1,
                         out_amax=self.dh1_amax)
        p["o"].dgrad_q(self.dh1, self.dh1q, self.dattn, amax=self.dh1_amax)  # into attention
        if side is None:
            self._qkv_dgrad(dq, dk, dv)
        else:
            main.wait_stream(side)
        pact_rmsnorm_bwd(self.xq1, self.gamma1, self.rstd1, self.dxn1, dres=self.dh1, dx=self.dx)
        return self.dx

    def _qkv_dgrad(self, dq, dk, dv):
        p = self.p
        p["q"].dgrad_q(dq, self.dqq, self.dxn1)
        p["k"].dgrad_q(dk, self.dkq, self.dxn1, accumulate=True)
        p["v"].dgrad_q(dv, self.dvq, self.dxn1, accumulate=True)

    @classmethod
    def from_workload(cls, d: dict, device) -> "DecoderProjectionStack":
        """Build the stack from host arrays: d holds x (for M), gamma1, gamma2, eps and
        projections q, k, v, o, gate_up, down with FP32 W [d_out, d_in], adapters A
        [d_in, r], B [r, d_out] (BF16 values) and alpha, r.  Weights are packed here."""
        def t32(a):
            return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)

        proj = {}
        for k in ("q", "k", "v", "o", "gate_up", "down"):
            p = d[k]
            proj[k] = LoraLinear(t32(p.W), t32(p.A).bfloat16(), t32(p.B).bfloat16(),
                                 float(p.alpha) / float(p.r), gate_up=(k == "gate_up"))
        return cls(d["x"].shape[0], proj, t32(d["gamma1"]).bfloat16(),
                   t32(d["gamma2"]).bfloat16(), float(d["eps"]))

    def gemm_flops(self) -> float:
        """2*M*N*K over the 12 frozen-projection GEMMs of one forward + dgrad pass (six
        projections, q, k, v, o, gate|up and down, each forward and input gradient)."""
        return 2.0 * sum(l.gemm_flops(self.m) for l in self.p.values())
