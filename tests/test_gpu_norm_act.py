"""GPU parity of the fused RMSNorm -> NVFP4 and SiLU-multiply -> NVFP4 kernels
(bit-exact codes, scales, per-tensor scales and the FP32 rstd statistic) and of
their backward kernels (within |gpu-ref| <= 8e-3|ref| + 2e-3 rms(ref))."""
import numpy as np
import pytest
import torch

import oracle as orc
from nvfp4_frozen_projection_gb300 import (pact_check_status, pact_rmsnorm_bwd,
                                           pact_rmsnorm_quant, pact_silu_mul_bwd,
                                           pact_silu_mul_quant)
from nvfp4_frozen_projection_gb300 import workloads as wl

from gpu_helpers import assert_close, assert_nvfp4_equal, bf16, host

pytestmark = pytest.mark.gpu


def _rms_case(x, gamma, eps=np.float32(1e-5)):
    yq, rstd = pact_rmsnorm_quant(bf16(x), bf16(gamma), float(eps))
    pact_check_status()
    ref_q, ref_rstd = orc.rmsnorm_quant(x, gamma, eps)
    got = rstd.cpu().numpy()
    assert got.view(np.uint32).tolist() == ref_rstd.view(np.uint32).tolist() or \
        np.array_equal(got.view(np.uint32), ref_rstd.view(np.uint32)), \
        f"rstd differs in {np.count_nonzero(got.view(np.uint32) != ref_rstd.view(np.uint32))} rows"
    assert_nvfp4_equal(yq, ref_q, f"rmsnorm {x.shape}")
    return yq, rstd, ref_q, ref_rstd


@pytest.mark.parametrize("shape", [(64, 256), (130, 2048), (1, 64), (257, 3072), (33, 4096),
                                   (9, 960)])
def test_rmsnorm_quant_bit_exact(shape):
    rng = np.random.default_rng(shape[0] * 31 + shape[1])
    x = wl.bf16_round(wl.student_t_unit_rms(rng, shape))
    gamma = wl.bf16_round(1.0 + wl.normal(rng, (shape[1],), 0.1))
    _rms_case(x, gamma)


def test_rmsnorm_quant_full_size_workloads():
    d = wl.attn1b()
    _rms_case(d["x"], d["gamma"])
    d5 = wl.layer3b()
    _rms_case(d5["x"], d5["gamma1"])


def _gateup(rng, M, I, std=1.1):
    return wl.bf16_round(wl.normal(rng, (M, 2 * I), std))


@pytest.mark.parametrize("M,I", [(64, 256), (130, 1024), (1, 64), (300, 960)])
def test_silu_mul_quant_bit_exact(M, I):
    rng = np.random.default_rng(M + I)
    gu = _gateup(rng, M, I)
    gu[0, :8] = [0.0, -0.0, 50.0, -50.0, 90.0, -90.0, 1e-30, -200.0]
    hq, gq, uq = pact_silu_mul_quant(bf16(gu))
    pact_check_status()
    rh, rg, ru = orc.silu_mul_quant(gu)
    assert_nvfp4_equal(hq, rh, "h")
    assert_nvfp4_equal(gq, rg, "gate")
    assert_nvfp4_equal(uq, ru, "up")


@pytest.mark.parametrize("case", ["wide", "tiny_rows", "tiny_tensor", "tiny_gate"])
def test_silu_mul_quant_adversarial(case):
    """Inputs that push the kernel's fast-value shortcut to its exact fallbacks:
    |gate| beyond 80, exact and signed zeros, products that underflow, blocks whose
    decode step is zero or subnormal, and a whole tensor of tiny values."""
    rng = np.random.default_rng({"wide": 11, "tiny_rows": 12, "tiny_tensor": 13,
                                 "tiny_gate": 14}[case])
    M, I = 257, 1024
    g = rng.uniform(-100.0, 100.0, (M, I)).astype(np.float32)
    u = rng.standard_normal((M, I)).astype(np.float32)
    u[rng.random((M, I)) < 0.1] = 0.0
    u[rng.random((M, I)) < 0.05] = -0.0
    g[rng.random((M, I)) < 0.05] = -0.0
    if case == "tiny_rows":
        u[::7] *= np.float32(1e-37)   # h of these rows lands far below the tensor's scale
        u[3::11] = np.float32(1e-38)
    if case == "tiny_tensor":
        u *= np.float32(1e-36)
    if case == "tiny_gate":
        # gate values near the bottom of the range against large up values: h stays
        # ordinary while g / (1 + exp(-g)) is tiny
        m = rng.random((M, I)) < 0.2
        g[m] = rng.choice(np.array([1e-20, -1e-25, 3e-30, -1e-38, 2e-39], np.float32), m.sum())
        u[m] = rng.choice(np.array([1e15, -3e20, 1e25, 7e30, -2e35], np.float32), m.sum())
    gu = wl.bf16_round(np.concatenate([g, u], axis=1))
    hq, gq, uq = pact_silu_mul_quant(bf16(gu))
    pact_check_status()
    rh, rg, ru = orc.silu_mul_quant(gu)
    assert_nvfp4_equal(hq, rh, "h " + case)
    assert_nvfp4_equal(gq, rg, "gate " + case)
    assert_nvfp4_equal(uq, ru, "up " + case)


def test_silu_mul_quant_full_size_and_amax_opt():
    """Workload 3's SiLU input shape [4096, 2 x 8192]; also the single-pass variant
    that takes precomputed amax values."""
    rng = np.random.default_rng(303)
    gu = _gateup(rng, 4096, 8192)
    g_dev = bf16(gu)
    hq, gq, uq = pact_silu_mul_quant(g_dev)
    rh, rg, ru = orc.silu_mul_quant(gu)
    assert_nvfp4_equal(hq, rh, "h full")
    assert_nvfp4_equal(gq, rg, "gate full")
    assert_nvfp4_equal(uq, ru, "up full")
    h = orc.silu_mul_fp32(gu)
    amax3 = torch.tensor([orc.amax(h), orc.amax(gu[:, :8192]), orc.amax(gu[:, 8192:])],
                         dtype=torch.float32, device="cuda")
    hq2, gq2, uq2 = pact_silu_mul_quant(g_dev, amax3=amax3)
    assert_nvfp4_equal(hq2, rh, "h amax_opt")
    assert_nvfp4_equal(uq2, ru, "up amax_opt")


@pytest.mark.parametrize("M,I", [(64, 256), (130, 1024), (4096, 8192)])
def test_silu_mul_bwd(M, I):
    rng = np.random.default_rng(M * 3 + I)
    gu = _gateup(rng, M, I, std=2.0)
    dh = wl.bf16_round(wl.normal(rng, (M, I), 1e-2))
    rh, rg, ru = orc.silu_mul_quant(gu)
    _, gq, uq = pact_silu_mul_quant(bf16(gu))
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    dgu = pact_silu_mul_bwd(gq, uq, bf16(dh), out_amax=amax)
    pact_check_status()
    ref = orc.silu_mul_bwd(rg, ru, dh)
    got = host(dgu)
    assert_close(got, ref, "silu bwd")
    assert float(amax.item()) == float(np.abs(got).max())


@pytest.mark.parametrize("M,H,with_res", [(64, 256, False), (130, 2048, True), (8192, 3072, True)])
def test_rmsnorm_bwd(M, H, with_res):
    rng = np.random.default_rng(M + H)
    x = wl.bf16_round(wl.student_t_unit_rms(rng, (M, H)))
    gamma = wl.bf16_round(1.0 + wl.normal(rng, (H,), 0.1))
    dy = wl.bf16_round(wl.normal(rng, (M, H), 1e-2))
    dres = wl.bf16_round(wl.normal(rng, (M, H), 1e-2)) if with_res else None
    yq, rstd = pact_rmsnorm_quant(bf16(x), bf16(gamma))
    amax = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    dx = pact_rmsnorm_bwd(yq, bf16(gamma), rstd, bf16(dy), None if dres is None else bf16(dres),
                          out_amax=amax)
    pact_check_status()
    ref_q, ref_rstd = orc.rmsnorm_quant(x, gamma)
    ref = orc.rmsnorm_bwd(ref_q, gamma, ref_rstd, dy, dres)
    got = host(dx)
    assert_close(got, ref, "rmsnorm bwd")
    # producer-epilogue amax: exactly the max |.| of the BF16 gradient written
    assert float(amax.item()) == float(np.abs(got).max())
