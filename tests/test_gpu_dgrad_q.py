"""The fused input-gradient entry (pact_lora_linear_dgrad_q: dY quantised to NVFP4
and its LoRA down-projection formed in one pass, then the NVFP4 dgrad GEMM).

It must reproduce the two-call path (pact_quant_nvfp4, then pact_lora_linear_dgrad)
byte for byte: codes, every scale byte of the padded atoms, g and the BF16 dX; and
its NVFP4 dY must equal the oracle's quantisation of the same tensor bit for bit.
Shapes cover one row, rows off the 128-row CTA and scale atom, every padded rank,
column counts whose 64-column chunks split unevenly over the CTAs of a cluster, a
given amax and the accumulate mode."""
import numpy as np
import pytest
import torch

import oracle as orc
from nvfp4_frozen_projection_gb300 import (NVFP4, pact_check_status, pact_lora_linear_dgrad,
                                           pact_lora_linear_dgrad_q, pact_pack_weight_bwd,
                                           pact_quant_nvfp4)
from nvfp4_frozen_projection_gb300 import workloads as wl

from gpu_helpers import assert_close, assert_nvfp4_equal, bf16, f32, host

pytestmark = pytest.mark.gpu


def _same_nvfp4(a: NVFP4, b: NVFP4, what):
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes), f"{what}: codes differ"
    assert torch.equal(a.sf, b.sf), f"{what}: scale bytes differ"
    assert torch.equal(a.g.view(torch.int32), b.g.view(torch.int32)), f"{what}: g differs"


@pytest.mark.parametrize("M,N,K,r,given_amax,acc", [
    (1, 64, 64, 1, False, False),
    (200, 256, 512, 16, False, False),
    (333, 192, 448, 24, True, True),
    (130, 512, 256, 32, False, True),
    (97, 320, 1024, 64, True, False),
    (512, 3072, 1024, 16, False, False),
    (300, 1600, 256, 16, False, True),  # 25 column chunks: an uneven 12 / 13 cluster split
])
def test_dgrad_q_matches_two_calls(M, N, K, r, given_amax, acc):
    rng = np.random.default_rng(M * 5 + N + K + r)
    dy = wl.bf16_round(rng.standard_normal((M, N)).astype(np.float32) * 0.01)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    A = wl.bf16_round(rng.standard_normal((K, r)).astype(np.float32) / np.sqrt(K))
    B = wl.bf16_round(rng.standard_normal((r, N)).astype(np.float32) * 0.1)
    prev = wl.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    wb = pact_pack_weight_bwd(f32(W))
    dyd, Ad, Bd = bf16(dy), bf16(A), bf16(B)
    amax = None
    if given_amax:
        amax = torch.tensor([float(np.abs(dy).max())], dtype=torch.float32, device="cuda")
    # two calls
    q_ref = pact_quant_nvfp4(dyd, amax=amax)
    dx_ref = pact_lora_linear_dgrad(q_ref, dyd, wb, Ad, Bd, 2.0,
                                    dx=bf16(prev) if acc else None, accumulate=acc)
    # fused; fill the output buffers with garbage first so that every byte is checked
    q = NVFP4.empty(M, N)
    q.codes.fill_(0xA5)
    q.sf.fill_(0x5A)
    q.g.fill_(-1.0)
    dx, q = pact_lora_linear_dgrad_q(dyd, wb, Ad, Bd, 2.0, amax=amax, dyq=q,
                                     dx=bf16(prev) if acc else None, accumulate=acc)
    pact_check_status()
    _same_nvfp4(q, q_ref, "dyq")
    assert torch.equal(dx, dx_ref), "dx differs from the two-call path"
    # and the quantisation is the oracle's, bit for bit
    assert_nvfp4_equal(q, orc.quantize(dy), "dyq vs oracle")


def test_dgrad_q_against_oracle_q3b():
    """Workload 2 (3B query projection, 4096 tokens): dX within the GEMM bound of the
    oracle on a seeded sample of rows."""
    d = wl.q3b()
    p = d["proj"]
    wb = pact_pack_weight_bwd(f32(p.W))
    dx, q = pact_lora_linear_dgrad_q(bf16(d["dy"]), wb, bf16(p.A), bf16(p.B), p.scale)
    pact_check_status()
    oq = orc.quantize(d["dy"])
    assert_nvfp4_equal(q, oq, "dyq")
    _, owb = orc.pack_weight(p.W)
    rows = np.unique(np.concatenate([[0, 4095], np.random.default_rng(5).choice(4096, 254,
                                                                               replace=False)]))
    ref = orc.lora_linear_dgrad(oq, d["dy"], owb, p.A, p.B, p.alpha, rows=rows)
    assert_close(host(dx)[rows], ref, "dgrad_q q3b")
