"""The fused gate|up forward with the SiLU statistics of its output
(pact_lora_linear_fwd_gate_up): its output must equal the plain forward's bit for
bit (the interleaved weight and adapter order only changes which tile computes a
column), its amax3 must equal max |silu(gate) up| by the oracle's exact FP32
recipe, max |gate| and max |up| of that output exactly, and the single-pass
SiLU-multiply quantisation fed with it must match the oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle as orc
from nvfp4_frozen_projection_gb300 import (pact_check_status, pact_lora_linear_fwd,
                                           pact_lora_linear_fwd_gate_up, pact_pack_weight_fwd,
                                           pact_pack_weight_fwd_gate_up, pact_quant_nvfp4,
                                           pact_silu_mul_quant)
from nvfp4_frozen_projection_gb300 import workloads as wl

from gpu_helpers import assert_nvfp4_equal, bf16, f32, host

pytestmark = pytest.mark.gpu


def _case(M, I, K, r, w_std, x_std=1.0, zero_rows=0, seed=0):
    rng = np.random.default_rng(seed + M + I + K)
    x = wl.bf16_round((rng.standard_normal((M, K)) * x_std).astype(np.float32))
    W = (rng.standard_normal((2 * I, K)) * w_std).astype(np.float32)
    A = wl.bf16_round((rng.standard_normal((K, r)) / np.sqrt(K)).astype(np.float32))
    B = wl.bf16_round((rng.standard_normal((r, 2 * I)) * 0.1).astype(np.float32))
    if zero_rows:  # some gate and up outputs exactly zero (frozen rows and adapter columns)
        W[:zero_rows] = 0.0
        W[I:I + zero_rows] = 0.0
        B[:, :zero_rows] = 0.0
        B[:, I:I + zero_rows] = 0.0
    return x, W, A, B


@pytest.mark.parametrize("M,I,K,r,w_std,x_std,zero_rows", [
    (200, 192, 256, 16, 0.05, 1.0, 0),    # ragged M, last 256-column tile partial (N = 384)
    (129, 128, 192, 32, 1.0, 4.0, 0),     # |gate| far above 80: outside the fast bound
    (300, 320, 320, 8, 0.05, 1.0, 40),    # exact zeros among the outputs (N = 640)
    (1024, 1024, 1024, 32, 0.02, 1.0, 0),
])
def test_gate_up_forward_and_amax3(M, I, K, r, w_std, x_std, zero_rows):
    x, W, A, B = _case(M, I, K, r, w_std, x_std, zero_rows)
    scale = 2.0
    xq = pact_quant_nvfp4(bf16(x))
    Wd = f32(W)
    y_ref = pact_lora_linear_fwd(xq, pact_pack_weight_fwd(Wd), bf16(A), bf16(B), scale)
    y, amax3 = pact_lora_linear_fwd_gate_up(xq, pact_pack_weight_fwd_gate_up(Wd), bf16(A),
                                            bf16(B), scale)
    pact_check_status()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), "output differs"
    gu = host(y)
    h = orc.silu_mul_fp32(gu)
    want = np.float32([np.abs(h).max(), np.abs(gu[:, :I]).max(), np.abs(gu[:, I:]).max()])
    got = amax3.cpu().numpy()
    assert got.view(np.uint32).tolist() == want.view(np.uint32).tolist(), (got, want)
    # one pass of SiLU-multiply with those amaxes: the oracle's bytes
    hq, gq, uq = pact_silu_mul_quant(y, amax3=amax3)
    pact_check_status()
    ref = orc.silu_mul_quant(gu)
    for t, r_, w in zip((hq, gq, uq), ref, ("h", "gate", "up")):
        assert_nvfp4_equal(t, r_, f"SiLU-multiply {w} with the GEMM's amaxes")


def test_interleaved_pack_is_a_row_permutation():
    """The gate|up forward pack holds the plain pack's rows, interleaved in groups of 32."""
    I, K = 96, 128
    W = (np.random.default_rng(3).standard_normal((2 * I, K)) * 0.02).astype(np.float32)
    a, b = pact_pack_weight_fwd(f32(W)), pact_pack_weight_fwd_gate_up(f32(W))
    pact_check_status()
    perm = np.concatenate([np.r_[32 * j:32 * j + 32, I + 32 * j:I + 32 * j + 32]
                           for j in range(I // 32)])
    assert np.array_equal(b.codes.cpu().numpy(), a.codes.cpu().numpy()[perm])
    sa = orc.unswizzle_scales(a.sf.cpu().numpy(), 2 * I, K // 16)
    sb = orc.unswizzle_scales(b.sf.cpu().numpy(), 2 * I, K // 16)
    assert np.array_equal(sb, sa[perm]) and a.g.item() == b.g.item()
