"""Oracle chains: the per-op oracle functions composed in the order the decoder
layer runs them.

TEST INFRASTRUCTURE ONLY (same rule as the rest of this package).

Source: "PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs", Figure 2 (the
decoder data flow: RMSNorm -> NVFP4 feeds the q, k and v projections (three
frozen weights, each with its own per-tensor scale), attention output feeds o, a
residual add, RMSNorm -> NVFP4 feeds the fused gate/up projection, SiLU-multiply
-> NVFP4 feeds down, a second residual add) and Table 7 (which tensors are kept in
NVFP4, which in BF16, and that gradients are BF16).

Every activation or gradient that the layer stores in BF16 between two operations
is rounded to BF16 here too (round_bf16), so both sides quantise the same kind of
value; the contractions themselves stay FP64.  The attention core and its backward
are not part of the stack: their output and the gradients they return are given
inputs.
"""
from __future__ import annotations

import numpy as np

from . import (lora_linear_dgrad, lora_linear_fwd, pack_weight, quantize, rmsnorm_bwd,
               rmsnorm_quant, silu_mul_bwd, silu_mul_quant)


def round_bf16(x) -> np.ndarray:
    """Round to the nearest BF16 value (8 significant bits, ties to even), from the
    definition of the format: values are split as m * 2^e with m in [0.5, 1), the
    mantissa m * 2^8 is rounded half-to-even, and values below the smallest normal
    (2^-126) round on the fixed subnormal grid 2^-133.  Returned as FP64."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)
    out = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    tiny = np.abs(x) < 2.0 ** -126
    if tiny.any():
        out[tiny] = np.ldexp(np.rint(np.ldexp(x[tiny], 133)), -133)
    return out


def _packs(projs: dict) -> dict:
    return {k: pack_weight(p.W) for k, p in projs.items()}


def attention_inputs(x, gamma, projs, dys, eps, packs=None) -> dict:
    """RMSNorm -> NVFP4 feeding the q, k, v projections, and the input gradient:
    the three dgrads accumulate into one BF16 buffer in the order q, k, v, then the
    RMSNorm backward.  projs: [q, k, v] objects with W, A, B, alpha."""
    packs = packs or [pack_weight(p.W) for p in projs]
    o = {}
    o["xq"], o["rstd"] = rmsnorm_quant(x, gamma, eps)
    o["y"] = [round_bf16(lora_linear_fwd(o["xq"], pk[0], p.A, p.B, p.alpha))
              for p, pk in zip(projs, packs)]
    o["dyq"] = [quantize(dy) for dy in dys]
    acc = None
    for p, pk, dyq, dy in zip(projs, packs, o["dyq"], dys):
        acc = round_bf16(lora_linear_dgrad(dyq, dy, pk[1], p.A, p.B, p.alpha, dx_prev=acc))
    o["dxn"] = acc
    o["dx"] = round_bf16(rmsnorm_bwd(o["xq"], gamma, o["rstd"], acc))
    return o


def mlp(x, gate_up, down, dy, packs=None) -> dict:
    """The MLP: NVFP4 x feeds the fused gate|up projection, SiLU-multiply -> NVFP4
    feeds down; backward: down dgrad, SiLU-multiply backward from the NVFP4 gate/up
    copies, one NVFP4 quantisation of d(gate|up), gate|up dgrad."""
    packs = packs or _packs({"gate_up": gate_up, "down": down})
    o = {}
    o["xq"] = quantize(x)
    o["gu"] = round_bf16(lora_linear_fwd(o["xq"], packs["gate_up"][0], gate_up.A, gate_up.B,
                                         gate_up.alpha))
    o["hq"], o["gq"], o["uq"] = silu_mul_quant(o["gu"])
    o["out"] = round_bf16(lora_linear_fwd(o["hq"], packs["down"][0], down.A, down.B,
                                          down.alpha))
    o["dyq"] = quantize(dy)
    o["dh"] = round_bf16(lora_linear_dgrad(o["dyq"], dy, packs["down"][1], down.A, down.B,
                                           down.alpha))
    o["dgu"] = round_bf16(silu_mul_bwd(o["gq"], o["uq"], o["dh"]))
    o["dguq"] = quantize(o["dgu"])
    o["dx"] = round_bf16(lora_linear_dgrad(o["dguq"], o["dgu"], packs["gate_up"][1], gate_up.A,
                                           gate_up.B, gate_up.alpha))
    return o


def decoder_layer(d: dict, packs=None) -> dict:
    """Forward and input-gradient pass of the decoder-layer projection stack.
    d holds x, attn, gamma1, gamma2, eps, the projections q, k, v, o, gate_up,
    down, and the incoming gradients dy (of the layer output) and dq, dk, dv (from
    the attention core into the q, k, v outputs).  The three input gradients of q,
    k and v accumulate into one BF16 buffer in that order.  Returns every
    intermediate."""
    names = ("q", "k", "v", "o", "gate_up", "down")
    P = {k: d[k] for k in names}
    packs = packs or _packs(P)

    def fwd(name, xq, residual=None):
        p = P[name]
        return round_bf16(lora_linear_fwd(xq, packs[name][0], p.A, p.B, p.alpha,
                                          residual=residual))

    def dgrad(name, gq, g, prev=None):
        p = P[name]
        return round_bf16(lora_linear_dgrad(gq, g, packs[name][1], p.A, p.B, p.alpha,
                                            dx_prev=prev))

    o = {}
    o["xq1"], o["rstd1"] = rmsnorm_quant(d["x"], d["gamma1"], d["eps"])
    for n in ("q", "k", "v"):
        o[n] = fwd(n, o["xq1"])
    o["attnq"] = quantize(d["attn"])
    o["h1"] = fwd("o", o["attnq"], residual=d["x"])
    o["xq2"], o["rstd2"] = rmsnorm_quant(o["h1"], d["gamma2"], d["eps"])
    o["gu"] = fwd("gate_up", o["xq2"])
    o["hq"], o["gq"], o["uq"] = silu_mul_quant(o["gu"])
    o["out"] = fwd("down", o["hq"], residual=o["h1"])
    o["dyq"] = quantize(d["dy"])
    o["dh"] = dgrad("down", o["dyq"], d["dy"])
    o["dgu"] = round_bf16(silu_mul_bwd(o["gq"], o["uq"], o["dh"]))
    o["dguq"] = quantize(o["dgu"])
    o["dxn2"] = dgrad("gate_up", o["dguq"], o["dgu"])
    o["dh1"] = round_bf16(rmsnorm_bwd(o["xq2"], d["gamma2"], o["rstd2"], o["dxn2"],
                                      dres=d["dy"]))
    o["dh1q"] = quantize(o["dh1"])
    o["dattn"] = dgrad("o", o["dh1q"], o["dh1"])
    o["dqq"], o["dkq"], o["dvq"] = (quantize(d[n]) for n in ("dq", "dk", "dv"))
    acc = dgrad("q", o["dqq"], d["dq"])
    acc = dgrad("k", o["dkq"], d["dk"], acc)
    o["dxn1"] = dgrad("v", o["dvq"], d["dv"], acc)
    o["dx"] = round_bf16(rmsnorm_bwd(o["xq1"], d["gamma1"], o["rstd1"], o["dxn1"],
                                     dres=o["dh1"]))
    return o
