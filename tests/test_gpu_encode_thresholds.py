"""GPU parity of the element encode q = e2m1(RN(x / t)) on quotients placed on and
beside the E2M1 rounding thresholds, where the GPU's certified products cannot
decide and its exact path must.  The per-tensor scale is set through the amax
argument, so that one BF16 value x0 (and its doubles) lands within a few FP32
steps of a threshold: t = RN(448 g) is tuned to x0 / m.  Every byte is compared
with the oracle; the same inputs are checked (on the host, with exact rationals)
to contain elements where multiplying by the rounded reciprocal would round to
another code."""
import numpy as np
import pytest
import torch

import oracle as orc
from exact_round import code_of_quotient
from nvfp4_frozen_projection_gb300 import workloads as wl
from nvfp4_frozen_projection_gb300 import (NVFP4, pact_check_status, pact_lora_linear_dgrad_q,
                                           pact_pack_weight_bwd, pact_pack_weight_fwd,
                                           pact_quant_nvfp4, pact_silu_mul_quant)

from gpu_helpers import assert_nvfp4_equal, bf16, dev, f32, host

pytestmark = pytest.mark.gpu


def _bf16(v):
    return np.float32(wl.bf16_round(np.float32([v]))[0])


def _scale_for(rng, x0, m0):
    """amax whose per-tensor scale g puts x0 / t, t = RN(448 g), within a few FP32
    steps of the threshold m0, preferring (when one is near) a g for which
    RN(x0 / t) and RN(x0 RN(1/t)) round to different E2M1 codes."""
    g0 = np.float32(x0 / m0 / 448.0)
    cands = []
    g = g0
    for _ in range(128):
        g = np.nextafter(g, np.float32(0))
    for _ in range(256):
        amax = np.float32(g * np.float32(2688.0))
        gg = orc.global_scale(amax)
        t = np.float32(448.0) * gg
        rcp = np.float32(1.0) / t
        apart = code_of_quotient(x0, t) != code_of_quotient(np.float32(x0 * rcp), np.float32(1.0))
        cands.append((amax, apart))
        g = np.nextafter(g, np.float32(np.inf))
    split = [c for c in cands if c[1]]
    if split and rng.random() < 0.8:
        return split[int(rng.integers(len(split)))][0], True
    return cands[int(rng.integers(len(cands)))][0], False


def _case(rng, rows=64, cols=128):
    """x [rows, cols] BF16 values and the amax to pass; every block holds a
    scale-448 element B and elements +-x0 * 2^j whose quotients sit at thresholds."""
    for _ in range(6):  # a few x0 until one has a splitting scale nearby
        m0 = float(rng.choice([0.25, 0.75, 1.25, 1.75]))
        x0 = _bf16(rng.uniform(1.0, 2.0))
        amax, split = _scale_for(rng, x0, m0)
        if split:
            break
    g = orc.global_scale(amax)                     # the scale both sides derive
    t = np.float32(448.0) * g
    B = _bf16(5.85 * float(t))                      # e4m3(B / 6g) = 448
    xb = wl.bf16_round((rng.standard_normal((rows, cols)) * 0.3 * float(t)).astype(np.float32))
    mults = [1.0, 2.0, 4.0] if m0 == 1.25 else ([1.0, 2.0] if m0 == 1.75 else [1.0])
    for r in range(rows):
        for b in range(cols // 16):
            xb[r, b * 16] = B if rng.random() < 0.5 else -B
            for i in range(1, 16):
                if rng.random() < 0.6:
                    v = x0 * float(rng.choice(mults))
                    xb[r, b * 16 + i] = -v if rng.random() < 0.4 else v
    return xb.astype(np.float32), amax


def test_quant_near_threshold_quotients():
    rng = np.random.default_rng(2024)
    apart = 0
    for trial in range(60):
        x, amax = _case(rng)
        xd = bf16(x)
        a = torch.tensor([float(amax)], dtype=torch.float32, device=dev())
        q = pact_quant_nvfp4(xd, amax=a)
        pact_check_status()
        ref = orc.quantize(x, g=orc.global_scale(amax))
        assert_nvfp4_equal(q, ref, f"near-threshold quant, trial {trial}")
        # discrimination: elements whose code differs under x * RN(1/t)
        t = np.float32(448.0) * ref.g
        rcp = np.float32(1.0) / t
        vals = np.unique(np.abs(x[:, :]))
        for v in vals:
            if v == 0:
                continue
            c_div = code_of_quotient(v, t)
            c_mul = code_of_quotient(np.float32(v * rcp), np.float32(1.0))
            apart += int(c_div != c_mul)
    assert apart > 0, "no input separated the two encode orders"


def test_fused_dy_quant_near_threshold_quotients():
    """The input-gradient entry's fused dY quantisation uses the same encode: its
    NVFP4 dY must match the oracle on the same threshold-straddling inputs."""
    rng = np.random.default_rng(77)
    K, r = 128, 16
    W = (rng.standard_normal((128, K)) * 0.02).astype(np.float32)
    wb = pact_pack_weight_bwd(f32(W))
    A = bf16((rng.standard_normal((K, r)) / np.sqrt(K)).astype(np.float32))
    Bm = bf16((rng.standard_normal((r, 128)) * 0.1).astype(np.float32))
    for trial in range(20):
        x, amax = _case(rng, rows=200, cols=128)
        dy = bf16(x)
        a = torch.tensor([float(amax)], dtype=torch.float32, device=dev())
        dyq = NVFP4.empty(200, 128, dev())
        pact_lora_linear_dgrad_q(dy, wb, A, Bm, 2.0, amax=a, dyq=dyq)
        pact_check_status()
        assert_nvfp4_equal(dyq, orc.quantize(x, g=orc.global_scale(amax)),
                           f"fused dY quant, trial {trial}")


def test_silu_gate_up_copies_near_threshold_quotients():
    """SiLU-multiply -> NVFP4 encodes its gate and up copies with the same element
    encode: threshold-straddling gate and up tensors (their amaxes passed in, h's
    exact amax from the oracle) must give the oracle's bytes for h, gate and up."""
    rng = np.random.default_rng(99)
    for trial in range(12):
        xg, ag = _case(rng, rows=64, cols=128)
        xu, au = _case(rng, rows=64, cols=128)
        gu = np.concatenate([xg, xu], axis=1)
        h = orc.silu_mul_fp32(gu)
        ah = np.float32(np.abs(h).max())
        a3 = torch.tensor([float(ah), float(ag), float(au)], dtype=torch.float32, device=dev())
        hq, gq, uq = pact_silu_mul_quant(bf16(gu), amax3=a3)
        pact_check_status()
        assert_nvfp4_equal(hq, orc.quantize(h, g=orc.global_scale(ah)), f"h, trial {trial}")
        assert_nvfp4_equal(gq, orc.quantize(xg, g=orc.global_scale(ag)), f"gate, trial {trial}")
        assert_nvfp4_equal(uq, orc.quantize(xu, g=orc.global_scale(au)), f"up, trial {trial}")


def test_weight_pack_near_threshold_quotients():
    """The frozen-weight packs encode with the same element rule: a weight whose 16x16
    tiles each hold a scale-448 element and threshold-straddling values, and whose
    amax (one element set to it) puts the per-tensor scale where the straddles are,
    must give the oracle's bytes in both layouts."""
    rng = np.random.default_rng(5)
    for trial in range(8):
        x, amax = _case(rng, rows=64, cols=128)
        W = x.copy()
        t = np.float32(448.0) * orc.global_scale(amax)
        for r0 in range(0, 64, 16):          # one scale-448 element per 16x16 tile
            for c0 in range(0, 128, 16):
                W[r0 + 1, c0 + 1] = _bf16(5.85 * float(t))
        W[0, 0] = amax                        # the tensor's amax, so g is the crafted one
        assert orc.global_scale(orc.amax(W)) == orc.global_scale(amax)
        rf, rb = orc.pack_weight(W)
        assert_nvfp4_equal(pact_pack_weight_fwd(f32(W)), rf, f"pack fwd, trial {trial}")
        assert_nvfp4_equal(pact_pack_weight_bwd(f32(W)), rb, f"pack bwd, trial {trial}")
        pact_check_status()
