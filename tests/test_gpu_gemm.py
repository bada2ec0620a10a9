"""GPU parity of the LoRA linear (NVFP4 tcgen05 GEMM + fused BF16 LoRA branch).

* Exact cases: host-constructed NVFP4 operands with g = 1, power-of-two scales and
  sparse integer adapters make every partial sum exactly representable in FP32, so
  the only rounding is the final BF16 cast and the GPU must equal it bit for bit.
  These pin the nibble order, the scale-factor layout and the MMA descriptors.
* Parity cases: seeded workload tensors quantised on both sides (bit-exact, see
  test_gpu_quant) and compared within |gpu-ref| <= 8e-3|ref| + 2e-3 rms(ref).
"""
import numpy as np
import pytest
import torch

import oracle as orc
from nvfp4_frozen_projection_gb300 import (pact_check_status, pact_lora_linear_dgrad,
                                           pact_lora_linear_fwd, pact_pack_weight_bwd,
                                           pact_pack_weight_fwd, pact_quant_nvfp4)
from nvfp4_frozen_projection_gb300 import workloads as wl

from gpu_helpers import assert_close, bf16, f32, host, nvfp4_to_device

pytestmark = pytest.mark.gpu


def _rand_q(rng, R, C, scales=(0x30, 0x38, 0x40)):
    codes = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    sc = rng.choice(np.array(scales, np.uint8), (R, C // 16))
    return orc.Q(codes, sc, np.float32(1.0), R, C)


def _sparse_pm1(rng, rows, cols, nnz_per_col):
    a = np.zeros((rows, cols), np.float32)
    for j in range(cols):
        idx = rng.choice(rows, nnz_per_col, replace=False)
        a[idx, j] = rng.choice([-1.0, 1.0], nnz_per_col)
    return a


def _bf16_of(exact):
    return torch.from_numpy(np.asarray(exact, np.float64)).float().to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("M,N,K,r", [(200, 256, 512, 16), (200, 384, 512, 16), (64, 256, 256, 8),
                                     (1, 64, 64, 1), (129, 320, 320, 24), (130, 512, 1024, 64)])
def test_fwd_exact_constructed(M, N, K, r):
    rng = np.random.default_rng(M * 7 + N + K + r)
    xq, wq = _rand_q(rng, M, K), _rand_q(rng, N, K)
    A = _sparse_pm1(rng, K, r, 2)                       # T = Xhat A stays BF16-exact
    B = rng.integers(-1, 2, (r, N)).astype(np.float32)
    ref = orc.lora_linear_fwd(xq, wq, A, B, alpha=float(r))  # scale alpha/r = 1
    y = pact_lora_linear_fwd(nvfp4_to_device(xq), nvfp4_to_device(wq), bf16(A), bf16(B), 1.0)
    pact_check_status()
    got = host(y)
    want = _bf16_of(ref)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}: " \
                          f"{[(got[tuple(i)], want[tuple(i)]) for i in bad[:4]]}"


@pytest.mark.parametrize("M,N,K,r,acc", [(200, 512, 256, 16, False), (130, 256, 384, 8, True),
                                         (64, 320, 128, 32, True)])
def test_dgrad_exact_constructed(M, N, K, r, acc):
    rng = np.random.default_rng(M + N * 3 + K + r)
    dyq = _rand_q(rng, M, N)
    wb = _rand_q(rng, K, N)
    dy = orc.dequant(dyq).astype(np.float32)            # BF16-exact
    A = rng.integers(-1, 2, (K, r)).astype(np.float32)
    B = _sparse_pm1(rng, N, r, 2).T.copy()              # U = dY B^T stays BF16-exact
    prev = rng.integers(-8, 9, (M, K)).astype(np.float32)
    ref = orc.lora_linear_dgrad(dyq, dy, wb, A, B, alpha=float(r), dx_prev=prev if acc else None)
    dx = bf16(prev) if acc else None
    out = pact_lora_linear_dgrad(nvfp4_to_device(dyq), bf16(dy), nvfp4_to_device(wb), bf16(A),
                                 bf16(B), 1.0, dx=dx, accumulate=acc)
    pact_check_status()
    got = host(out)
    want = _bf16_of(ref)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:4].tolist()}"


def _layer(d_x, proj, dy=None, rows=None):
    """Run fwd (+ dgrad) on the GPU and the oracle from the same seeded inputs."""
    x = bf16(d_x)
    W = f32(proj.W)
    A, B = bf16(proj.A), bf16(proj.B)
    xq = pact_quant_nvfp4(x)
    wf, wb = pact_pack_weight_fwd(W), pact_pack_weight_bwd(W)
    y = pact_lora_linear_fwd(xq, wf, A, B, proj.scale)
    out = {"y": host(y)}
    oxq = orc.quantize(d_x)
    owf, owb = orc.pack_weight(proj.W)
    out["y_ref"] = orc.lora_linear_fwd(oxq, owf, proj.A, proj.B, proj.alpha, rows=rows)
    if dy is not None:
        dyb = bf16(dy)
        dyq = pact_quant_nvfp4(dyb)
        dx = pact_lora_linear_dgrad(dyq, dyb, wb, A, B, proj.scale)
        out["dx"] = host(dx)
        out["dx_ref"] = orc.lora_linear_dgrad(orc.quantize(dy), dy, owb, proj.A, proj.B,
                                              proj.alpha, rows=rows)
    pact_check_status()
    return out


def test_parity_tiny_workload():
    d = wl.tiny()
    o = _layer(d["x"], d["proj"], d["dy"])
    assert_close(o["y"], o["y_ref"], "fwd")
    assert_close(o["dx"], o["dx_ref"], "dgrad")


def test_parity_q3b_full_size_sampled_rows():
    """Workload 2 at full size; oracle on a seeded sample of 512 rows (first and
    last included), every column."""
    d = wl.q3b()
    rng = np.random.default_rng(2002)
    rows = np.unique(np.concatenate([[0, 4095], rng.choice(4096, 510, replace=False)]))
    o = _layer(d["x"], d["proj"], d["dy"], rows=rows)
    assert_close(o["y"][rows], o["y_ref"], "fwd q3b")
    assert_close(o["dx"][rows], o["dx_ref"], "dgrad q3b")


def test_lora_only_and_base_only():
    """W = 0 leaves the LoRA branch alone; B = 0 leaves the frozen product alone."""
    d = wl.tiny()
    p = d["proj"]
    for W, B in ((np.zeros_like(p.W), p.B), (p.W, np.zeros_like(p.B))):
        x = bf16(d["x"])
        y = pact_lora_linear_fwd(pact_quant_nvfp4(x), pact_pack_weight_fwd(f32(W)), bf16(p.A),
                                 bf16(B), p.scale)
        owf, _ = orc.pack_weight(W)
        ref = orc.lora_linear_fwd(orc.quantize(d["x"]), owf, p.A, B, p.alpha)
        assert_close(host(y), ref, "special case")


def test_residual_and_out_amax():
    d = wl.tiny()
    p = d["proj"]
    rng = np.random.default_rng(11)
    res = wl.bf16_round(rng.standard_normal((64, 256)).astype(np.float32))
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    x = bf16(d["x"])
    y = pact_lora_linear_fwd(pact_quant_nvfp4(x), pact_pack_weight_fwd(f32(p.W)), bf16(p.A),
                             bf16(p.B), p.scale, residual=bf16(res), out_amax=amax)
    owf, _ = orc.pack_weight(p.W)
    ref = orc.lora_linear_fwd(orc.quantize(d["x"]), owf, p.A, p.B, p.alpha, residual=res)
    assert_close(host(y), ref, "residual")
    assert float(amax.item()) == float(np.abs(host(y)).max())


@pytest.mark.parametrize("M,N,K,r", [(1, 64, 64, 4), (333, 192, 448, 12), (256, 2048, 512, 16)])
def test_parity_odd_shapes(M, N, K, r):
    rng = np.random.default_rng(M + N + K)
    x = wl.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    p = wl.make_proj(rng, "p", K, N, r, 2.0 * r, w_std=0.05)
    dy = wl.bf16_round(rng.standard_normal((M, N)).astype(np.float32) * 0.1)
    o = _layer(x, p, dy)
    assert_close(o["y"], o["y_ref"], "fwd odd")
    assert_close(o["dx"], o["dx_ref"], "dgrad odd")
