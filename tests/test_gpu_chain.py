"""The decoder-layer projection stack (workload 5), its MLP (workload 3) and its
attention-input block (workload 4) run on the GPU, each at a small size (every
row compared) and at the full benchmarked size (M = 8192, 4096 and 26624; 512
seeded rows plus the tile-edge rows compared for row-wise outputs, every byte for
NVFP4 outputs).

Every stage is checked against the oracle fed with the GPU's own upstream tensors
(tests/stage_checks.py), so each is held to its per-op bar: NVFP4 codes, scales, g
and the RMSNorm statistic bit-exact, GEMM and backward outputs within
|gpu - ref| <= 8e-3 |ref| + 2e-3 rms(ref).  At full size the GEMMs take every path
the benchmark takes, the banded tile order for A operands above 32 MiB (gate|up
input gradient, down forward) included.  The q, k and v input gradients, which
accumulate into one buffer, are re-run one at a time so that each accumulation
step is compared from the GPU's own previous buffer.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import nvfp4_frozen_projection_gb300 as pk
from nvfp4_frozen_projection_gb300 import workloads as wl
from nvfp4_frozen_projection_gb300.stack import DecoderProjectionStack, LoraLinear

from gpu_helpers import host
from stage_checks import (check_dgrad, check_fwd, check_quant, check_rmsnorm_bwd,
                          check_rmsnorm_quant, check_silu_bwd, check_silu_quant, sample_rows)

pytestmark = pytest.mark.gpu

PROJS = ("q", "k", "v", "o", "gate_up", "down")
LAYER_SIZES = {"small": dict(m=320, hidden=512, kv=128, inter=1024), "full": {}}


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).bfloat16().cuda()


def _lin(p):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    return LoraLinear(t(p.W), t(p.A).bfloat16(), t(p.B).bfloat16(), p.scale)


# ------------------------------------------------------------------ decoder layer
@pytest.fixture(scope="module", params=sorted(LAYER_SIZES))
def layer(request):
    d = wl.layer3b(**LAYER_SIZES[request.param])
    st = DecoderProjectionStack.from_workload(d, "cuda")
    ins = {n: _dev(d[n]) for n in ("x", "attn", "dy", "dq", "dk", "dv")}
    st.forward(ins["x"], ins["attn"])
    st.backward(ins["dy"], ins["dq"], ins["dk"], ins["dv"])
    torch.cuda.synchronize()
    pk.pact_check_status()
    packs = {n: orc.pack_weight(d[n].W) for n in PROJS}
    yield d, packs, st, ins, sample_rows(st.m)
    del st
    torch.cuda.empty_cache()


def test_layer_forward_stages(layer):
    d, packs, st, ins, rows = layer
    gamma1, gamma2, eps = d["gamma1"], d["gamma2"], d["eps"]
    check_rmsnorm_quant("xq1", st.xq1, st.rstd1, ins["x"], gamma1, eps)
    for n in ("q", "k", "v"):
        check_fwd(n, getattr(st, n), st.xq1, d[n], packs[n][0], rows)
    check_quant("attnq", st.attnq, ins["attn"])
    check_fwd("o (+ residual x)", st.h1, st.attnq, d["o"], packs["o"][0], rows,
              residual=ins["x"])
    check_rmsnorm_quant("xq2", st.xq2, st.rstd2, st.h1, gamma2, eps)
    check_fwd("gate|up", st.gu, st.xq2, d["gate_up"], packs["gate_up"][0], rows)
    # the gate|up GEMM's epilogue amaxes, which the one-pass SiLU-multiply used
    gu = host(st.gu)
    inter = gu.shape[1] // 2
    want = np.float32([np.abs(orc.silu_mul_fp32(gu)).max(), np.abs(gu[:, :inter]).max(),
                       np.abs(gu[:, inter:]).max()])
    assert st.gu_amax3.cpu().numpy().view(np.uint32).tolist() == want.view(np.uint32).tolist()
    check_silu_quant("SiLU-multiply", st.hq, st.gq, st.uq, st.gu)
    check_fwd("down (+ residual h1)", st.out, st.hq, d["down"], packs["down"][0], rows,
              residual=st.h1)


def test_layer_backward_stages(layer):
    d, packs, st, ins, rows = layer
    gamma1, gamma2 = d["gamma1"], d["gamma2"]
    check_quant("dY", st.dyq, ins["dy"])
    check_dgrad("down", st.dh, st.dyq, ins["dy"], d["down"], packs["down"][1], rows)
    check_silu_bwd("SiLU-multiply", st.dgu, st.gq, st.uq, st.dh, rows, amax=st.dgu_amax)
    check_quant("d(gate|up)", st.dguq, st.dgu, amax=st.dgu_amax)
    check_dgrad("gate|up", st.dxn2, st.dguq, st.dgu, d["gate_up"], packs["gate_up"][1], rows)
    check_rmsnorm_bwd("RMSNorm 2 (+ dres dy)", st.dh1, st.xq2, gamma2, st.rstd2, st.dxn2, rows,
                      dres=ins["dy"], amax=st.dh1_amax)
    check_quant("dh1", st.dh1q, st.dh1, amax=st.dh1_amax)
    check_dgrad("o", st.dattn, st.dh1q, st.dh1, d["o"], packs["o"][1], rows)
    for n, q in (("dq", st.dqq), ("dk", st.dkq), ("dv", st.dvq)):
        check_quant(n, q, ins[n])
    check_rmsnorm_bwd("RMSNorm 1 (+ dres dh1)", st.dx, st.xq1, gamma1, st.rstd1, st.dxn1, rows,
                      dres=st.dh1)


def _qkv_accumulation(lins, packs, projs, dyqs, dys, rows, want):
    """Re-run the q, k, v input gradients one call at a time: each accumulation step
    is compared from the GPU's own previous buffer, and the final buffer must be the
    one the stack produced, bit for bit."""
    buf = torch.empty_like(want)
    prev = None
    for i, (l, pkb, p, dyq, dy) in enumerate(zip(lins, packs, projs, dyqs, dys)):
        l.dgrad(dyq, dy, buf, accumulate=i > 0)
        torch.cuda.synchronize()
        check_dgrad(f"{p.name} (accumulate={i > 0})", buf, dyq, dy, p, pkb, rows, dx_prev=prev)
        prev = buf.clone()
    assert torch.equal(buf, want), "re-run accumulation differs from the stack's"


def test_layer_qkv_accumulation(layer):
    d, packs, st, ins, rows = layer
    names = ("q", "k", "v")
    _qkv_accumulation([st.p[n] for n in names], [packs[n][1] for n in names],
                      [d[n] for n in names], [st.dqq, st.dkq, st.dvq],
                      [ins["dq"], ins["dk"], ins["dv"]], rows, st.dxn1)


# ------------------------------------------------------------------ MLP block
@pytest.mark.parametrize("m", [320, 4096])
def test_mlp_stages(m):
    kw = dict(m=320, hidden=512, inter=1024) if m == 320 else {}
    d = wl.mlp3b(**kw)
    gate_up, down = _lin(d["gate_up"]), _lin(d["down"])
    pg, pd = orc.pack_weight(d["gate_up"].W), orc.pack_weight(d["down"].W)
    x, dy = _dev(d["x"]), _dev(d["dy"])
    xq = pk.pact_quant_nvfp4(x)
    gu = pk.pact_lora_linear_fwd(xq, gate_up.w_fwd, gate_up.A, gate_up.B, gate_up.scale)
    hq, gq, uq = pk.pact_silu_mul_quant(gu)
    out = pk.pact_lora_linear_fwd(hq, down.w_fwd, down.A, down.B, down.scale)
    dh, dyq = pk.pact_lora_linear_dgrad_q(dy, down.w_bwd, down.A, down.B, down.scale)
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    dgu = pk.pact_silu_mul_bwd(gq, uq, dh, out_amax=amax)
    dx, dguq = pk.pact_lora_linear_dgrad_q(dgu, gate_up.w_bwd, gate_up.A, gate_up.B,
                                           gate_up.scale, amax=amax)
    pk.pact_check_status()
    rows = sample_rows(m)
    check_quant("x", xq, x)
    check_fwd("gate|up", gu, xq, d["gate_up"], pg[0], rows)
    check_silu_quant("SiLU-multiply", hq, gq, uq, gu)
    check_fwd("down", out, hq, d["down"], pd[0], rows)
    check_quant("dY", dyq, dy)
    check_dgrad("down", dh, dyq, dy, d["down"], pd[1], rows)
    check_silu_bwd("SiLU-multiply", dgu, gq, uq, dh, rows, amax=amax)
    check_quant("d(gate|up)", dguq, dgu, amax=amax)
    check_dgrad("gate|up", dx, dguq, dgu, d["gate_up"], pg[1], rows)


# ------------------------------------------------------------ attention inputs
@pytest.mark.parametrize("m", [320, 26624])
def test_attention_input_stages(m):
    kw = dict(m=320, hidden=512, kv=128) if m == 320 else {}
    d = wl.attn1b(**kw)
    lins = [_lin(p) for p in d["projs"]]
    packs = [orc.pack_weight(p.W) for p in d["projs"]]
    x = _dev(d["x"])
    gamma = torch.from_numpy(np.ascontiguousarray(d["gamma"], np.float32)).cuda().bfloat16()
    xq, rstd = pk.pact_rmsnorm_quant(x, gamma, float(d["eps"]))
    ys = [l.forward(xq, torch.empty(m, l.d_out, dtype=torch.bfloat16, device="cuda"))
          for l in lins]
    dys = [_dev(a) for a in d["dys"]]
    dyqs = [pk.pact_quant_nvfp4(t) for t in dys]
    dn = torch.empty(m, x.shape[1], dtype=torch.bfloat16, device="cuda")
    for i, (l, dy, dyq) in enumerate(zip(lins, dys, dyqs)):
        l.dgrad(dyq, dy, dn, accumulate=i > 0)
    dx = pk.pact_rmsnorm_bwd(xq, gamma, rstd, dn)
    pk.pact_check_status()
    rows = sample_rows(m)
    check_rmsnorm_quant("x", xq, rstd, x, d["gamma"], d["eps"])
    for p, pw, y in zip(d["projs"], packs, ys):
        check_fwd(p.name, y, xq, p, pw[0], rows)
    for p, dyq, dy in zip(d["projs"], dyqs, dys):
        check_quant("d" + p.name, dyq, dy)
    _qkv_accumulation(lins, [pw[1] for pw in packs], d["projs"], dyqs, dys, rows, dn)
    check_rmsnorm_bwd("RMSNorm", dx, xq, d["gamma"], rstd, dn, rows)
