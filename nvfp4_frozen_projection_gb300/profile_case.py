"""One libpact operation on seeded inputs, repeated a few times, for a profiler.

    python -m nvfp4_frozen_projection_gb300.profile_case <case> [--m M] [--reps R]

Cases (M = tokens; the other sizes are the Llama-3B layer's):
  gemm-gate-up-dgrad  dX = dY W (NVFP4, K = 2 x 8192) + LoRA term, out 3072 wide
  gemm-gate-up-fwd    Y = X W^T (NVFP4, 3072 -> 2 x 8192) + LoRA term
  gemm-gate-up-stats  the same GEMM on the interleaved gate|up weight, its epilogue
                      also forming the SiLU-multiply amaxes (pact_lora_linear_fwd_gate_up)
  quant               NVFP4 quantisation of a BF16 [M, 3072] tensor
  silu                SiLU-multiply -> NVFP4 of a BF16 [M, 2 x 8192] tensor
  silu-amax3          the same in one pass, with the three amaxes the gate|up forward
                      GEMM emits (the GEMM runs once, before the repetitions)
  lora-down-fwd       the q projection's forward (down-projection + GEMM)
  gemm-o-fwd          the o projection's forward: the same GEMM plus the residual add
  dgrad-q-gate-up     the fused gate|up input gradient (dY quantised inside the LoRA
                      down-projection, then the GEMM): pact_lora_linear_dgrad_q
  dgrad-q-q           the same for the q projection (3072 -> 3072, r = 16)
  adapter-grad-q      dA, dB of the q projection (3072 -> 3072, r = 16)
  adapter-grad-gate-up  dA, dB of the fused gate|up projection (3072 -> 2 x 8192, r = 32)
  rmsnorm             RMSNorm -> NVFP4 of a BF16 [M, 3072] tensor (statistic and encode)
  rmsnorm-bwd         RMSNorm backward of a [M, 3072] NVFP4 output, with a residual gradient
  silu-bwd            SiLU-multiply backward from [M, 8192] NVFP4 gate/up copies
  pack-weight         forward and backward NVFP4 packs of the gate|up weight [2 x 8192, 3072]

The default M (4096) keeps the inputs of the SiLU, GEMM and weight-pack cases above
the 129 MB L2 and every case's device memory under 1 GB, the size a full ncu capture
wants; the [M, 3072] cases (quant, rmsnorm, rmsnorm-bwd) need --m 32768 (16384 for
rmsnorm-bwd) for their inputs to exceed the L2.  Each run exits 0
only if the library's status word is clear.
"""
from __future__ import annotations

import argparse

import torch

from . import (pact_check_status, pact_lora_adapter_grad, pact_lora_linear_dgrad,
               pact_lora_linear_dgrad_q, pact_lora_linear_fwd_gate_up,
               pact_pack_weight_fwd_gate_up,
               pact_lora_linear_fwd, pact_pack_weight_bwd, pact_pack_weight_fwd,
               pact_quant_nvfp4, pact_rmsnorm_bwd, pact_rmsnorm_quant, pact_silu_mul_bwd,
               pact_silu_mul_quant)

HIDDEN, INTER = 3072, 8192


def _lora(d_in, d_out, r, dev, gen):
    W = torch.randn(d_out, d_in, device=dev, generator=gen) * 0.02
    A = (torch.randn(d_in, r, device=dev, generator=gen) / d_in ** 0.5).bfloat16()
    B = (torch.randn(r, d_out, device=dev, generator=gen) * 0.1).bfloat16()
    return W, A, B


def run(case: str, m: int, reps: int) -> None:
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    if case == "gemm-gate-up-dgrad":
        W, A, B = _lora(HIDDEN, 2 * INTER, 32, dev, gen)
        wb = pact_pack_weight_bwd(W)
        dy = (torch.randn(m, 2 * INTER, device=dev, generator=gen) * 0.01).bfloat16()
        dyq = pact_quant_nvfp4(dy)
        dx = torch.empty(m, HIDDEN, dtype=torch.bfloat16, device=dev)
        for _ in range(reps):
            pact_lora_linear_dgrad(dyq, dy, wb, A, B, 2.0, dx=dx)
    elif case in ("dgrad-q-gate-up", "dgrad-q-q"):
        n_out, r = (2 * INTER, 32) if case == "dgrad-q-gate-up" else (HIDDEN, 16)
        W, A, B = _lora(HIDDEN, n_out, r, dev, gen)
        wb = pact_pack_weight_bwd(W)
        dy = (torch.randn(m, n_out, device=dev, generator=gen) * 0.01).bfloat16()
        amax = dy.float().abs().max().reshape(1)
        dx = torch.empty(m, HIDDEN, dtype=torch.bfloat16, device=dev)
        dyq = None
        for _ in range(reps):
            dx, dyq = pact_lora_linear_dgrad_q(dy, wb, A, B, 2.0, amax=amax, dyq=dyq, dx=dx)
    elif case in ("gemm-gate-up-fwd", "lora-down-fwd", "gemm-o-fwd"):
        n_out = 2 * INTER if case == "gemm-gate-up-fwd" else HIDDEN
        r = 32 if case == "gemm-gate-up-fwd" else 16
        W, A, B = _lora(HIDDEN, n_out, r, dev, gen)
        wf = pact_pack_weight_fwd(W)
        x = torch.randn(m, HIDDEN, device=dev, generator=gen).bfloat16()
        xq = pact_quant_nvfp4(x)
        res = x if case == "gemm-o-fwd" else None
        y = torch.empty(m, n_out, dtype=torch.bfloat16, device=dev)
        for _ in range(reps):
            pact_lora_linear_fwd(xq, wf, A, B, 2.0, residual=res, y=y)
    elif case in ("adapter-grad-q", "adapter-grad-gate-up"):
        n_out, r = (HIDDEN, 16) if case == "adapter-grad-q" else (2 * INTER, 32)
        _, A, B = _lora(HIDDEN, n_out, r, dev, gen)
        x = torch.randn(m, HIDDEN, device=dev, generator=gen).bfloat16()
        xq = pact_quant_nvfp4(x)
        dy = (torch.randn(m, n_out, device=dev, generator=gen) * 0.01).bfloat16()
        dA = torch.empty(HIDDEN, r, dtype=torch.float32, device=dev)
        dB = torch.empty(r, n_out, dtype=torch.float32, device=dev)
        for _ in range(reps):
            pact_lora_adapter_grad(xq, dy, A, B, 2.0, dA=dA, dB=dB)
    elif case == "quant":
        x = torch.randn(m, HIDDEN, device=dev, generator=gen).bfloat16()
        q = pact_quant_nvfp4(x)
        for _ in range(reps):
            pact_quant_nvfp4(x, out=q)
    elif case == "silu":
        gu = torch.randn(m, 2 * INTER, device=dev, generator=gen).bfloat16()
        outs = pact_silu_mul_quant(gu)
        for _ in range(reps):
            pact_silu_mul_quant(gu, outs=outs)
    elif case == "gemm-gate-up-stats":
        W, A, B = _lora(HIDDEN, 2 * INTER, 32, dev, gen)
        wg = pact_pack_weight_fwd_gate_up(W)
        xq = pact_quant_nvfp4(torch.randn(m, HIDDEN, device=dev, generator=gen).bfloat16())
        y = torch.empty(m, 2 * INTER, dtype=torch.bfloat16, device=dev)
        a3 = torch.empty(3, dtype=torch.float32, device=dev)
        for _ in range(reps):
            pact_lora_linear_fwd_gate_up(xq, wg, A, B, 2.0, y=y, amax3=a3)
    elif case == "silu-amax3":
        W, A, B = _lora(HIDDEN, 2 * INTER, 32, dev, gen)
        x = torch.randn(m, HIDDEN, device=dev, generator=gen).bfloat16()
        gu, amax3 = pact_lora_linear_fwd_gate_up(pact_quant_nvfp4(x),
                                                 pact_pack_weight_fwd_gate_up(W), A, B, 2.0)
        outs = pact_silu_mul_quant(gu, amax3=amax3)
        for _ in range(reps):
            pact_silu_mul_quant(gu, amax3=amax3, outs=outs)
    elif case == "rmsnorm":
        x = torch.randn(m, HIDDEN, device=dev, generator=gen).bfloat16()
        gamma = (1.0 + 0.1 * torch.randn(HIDDEN, device=dev, generator=gen)).bfloat16()
        yq, rstd = pact_rmsnorm_quant(x, gamma)
        for _ in range(reps):
            pact_rmsnorm_quant(x, gamma, out=yq, rstd=rstd)
    elif case == "rmsnorm-bwd":
        x = torch.randn(m, HIDDEN, device=dev, generator=gen).bfloat16()
        gamma = (1.0 + 0.1 * torch.randn(HIDDEN, device=dev, generator=gen)).bfloat16()
        yq, rstd = pact_rmsnorm_quant(x, gamma)
        dy = (torch.randn(m, HIDDEN, device=dev, generator=gen) * 0.01).bfloat16()
        dres = (torch.randn(m, HIDDEN, device=dev, generator=gen) * 0.01).bfloat16()
        dx = torch.empty_like(dy)
        amax = torch.empty(1, dtype=torch.float32, device=dev)
        for _ in range(reps):
            pact_rmsnorm_bwd(yq, gamma, rstd, dy, dres=dres, dx=dx, out_amax=amax)
    elif case == "silu-bwd":
        gu = torch.randn(m, 2 * INTER, device=dev, generator=gen).bfloat16()
        _, gq, uq = pact_silu_mul_quant(gu)
        dh = (torch.randn(m, INTER, device=dev, generator=gen) * 0.01).bfloat16()
        dgu = torch.empty_like(gu)
        amax = torch.empty(1, dtype=torch.float32, device=dev)
        for _ in range(reps):
            pact_silu_mul_bwd(gq, uq, dh, dgateup=dgu, out_amax=amax)
    elif case == "pack-weight":
        W = torch.randn(2 * INTER, HIDDEN, device=dev, generator=gen) * 0.02
        wf, wb = pact_pack_weight_fwd(W), pact_pack_weight_bwd(W)
        for _ in range(reps):
            pact_pack_weight_fwd(W, out=wf)
            pact_pack_weight_bwd(W, out=wb)
    else:
        raise SystemExit(f"unknown case {case!r}")
    torch.cuda.synchronize()
    pact_check_status()


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--m", type=int, default=4096)
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args()
    run(a.case, a.m, a.reps)
    print("ok")


if __name__ == "__main__":
    main()
