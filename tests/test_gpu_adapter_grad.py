"""GPU parity of the LoRA adapter gradients dA = s Xhat^T (dY B^T), dB = s (Xhat A)^T dY.

* Exact cases: host-constructed NVFP4 inputs (power-of-two scales, per-tensor g a
  power of two), sparse adapters whose nonzeros include 1 + 2^-7 (so that dY B^T and
  Xhat A need more than BF16's 8 significant bits and the low half of their hi|lo
  carry is exercised) and power-of-two LoRA scales.  Every intermediate is then
  representable and every sum stays below 2^24 units of its granularity, so the
  FP32 results must equal the FP64 oracle bit for bit.  Shapes cover one row, row
  counts that leave a ragged 32-row round and a ragged row split, column counts that
  are not a multiple of the 128-column tile, and every padded rank (16, 32, 64).
* Parity cases: seeded workload tensors (the GPU quantises its own input, the oracle
  its own; the two agree bit for bit, see test_gpu_quant), compared element by
  element with the common bound |gpu-ref| <= 8e-3|ref| + 2e-3 rms(ref), and in
  relative RMS error with a bound of 2^-12.  That bound follows from the arithmetic:
  the hi|lo pair carries dY B^T and Xhat A to about 2^-16 relative, the products with
  Xhat and dY are exact in FP32 and FP32 accumulation adds a random-walk error of
  order 2^-24 sqrt(M); dropping the low half would give about 2^-10.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from nvfp4_frozen_projection_gb300 import (pact_check_status, pact_lora_adapter_grad,
                                           pact_quant_nvfp4)
from nvfp4_frozen_projection_gb300 import workloads as wl

from gpu_helpers import assert_close, bf16, host, nvfp4_to_device

pytestmark = pytest.mark.gpu

REL_RMS_BOUND = 2.0 ** -12


def _rand_q(rng, R, C, g=1.0):
    codes = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    sc = np.full((R, C // 16), 0x30, np.uint8)  # block scale 0.5: |Xhat| <= 3 g
    return orc.Q(codes, sc, np.float32(g), R, C)


def _sparse(rng, rows, cols, nnz_per_col):
    """nnz_per_col nonzeros per column, each +-1 or +-(1 + 2^-7)."""
    a = np.zeros((rows, cols), np.float32)
    for j in range(cols):
        idx = rng.choice(rows, nnz_per_col, replace=False)
        a[idx, j] = rng.choice([-1.0, 1.0], nnz_per_col) * rng.choice([1.0, 1.0 + 2.0 ** -7],
                                                                       nnz_per_col)
    return a


def _rel_rms(got, ref):
    ref = np.asarray(ref, np.float64)
    return float(np.sqrt(np.mean((got - ref) ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-300))


@pytest.mark.parametrize("M,N,K,r,scale,g", [
    (1, 64, 64, 1, 1.0, 1.0),
    (31, 128, 64, 8, 1.0, 1.0),
    (200, 256, 512, 16, 1.0, 1.0),
    (333, 192, 448, 24, 2.0, 0.5),
    (400, 512, 256, 32, 0.5, 2.0),
    (130, 320, 1024, 64, 1.0, 0.25),
    (97, 64, 192, 40, 4.0, 1.0),
])
def test_adapter_grad_exact_constructed(M, N, K, r, scale, g):
    rng = np.random.default_rng(M * 13 + N + K * 3 + r)
    xq = _rand_q(rng, M, K, g)
    dyq = _rand_q(rng, M, N)
    dy = orc.dequant(dyq).astype(np.float32)       # BF16-exact, |dY| <= 3
    A = _sparse(rng, K, r, 2)
    B = _sparse(rng, N, r, 2).T.copy()
    dA_ref, dB_ref = orc.lora_adapter_grad(xq, dy, A, B, alpha=scale * r)
    dA, dB = pact_lora_adapter_grad(nvfp4_to_device(xq), bf16(dy), bf16(A), bf16(B), scale)
    pact_check_status()
    for name, got, want in (("dA", host(dA), dA_ref), ("dB", host(dB), dB_ref)):
        want32 = want.astype(np.float32)
        assert np.array_equal(want32.astype(np.float64), want), f"{name}: case not FP32-exact"
        bad = np.argwhere(got != want32)
        assert bad.size == 0, f"{name}: {len(bad)} mismatches, first {bad[:4].tolist()}: " \
                              f"{[(got[tuple(i)], want32[tuple(i)]) for i in bad[:4]]}"


def test_adapter_grad_zero_inputs():
    """dY = 0 gives dA = dB = 0; so does X = 0 (every code zero)."""
    rng = np.random.default_rng(5)
    M, N, K, r = 96, 128, 256, 16
    A = wl.bf16_round(rng.standard_normal((K, r)).astype(np.float32))
    B = wl.bf16_round(rng.standard_normal((r, N)).astype(np.float32))
    x = wl.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    dA, dB = pact_lora_adapter_grad(pact_quant_nvfp4(bf16(x)), bf16(np.zeros((M, N))), bf16(A),
                                    bf16(B), 2.0)
    pact_check_status()
    assert not host(dA).any() and not host(dB).any()
    dy = wl.bf16_round(rng.standard_normal((M, N)).astype(np.float32))
    dA, dB = pact_lora_adapter_grad(pact_quant_nvfp4(bf16(np.zeros((M, K)))), bf16(dy), bf16(A),
                                    bf16(B), 2.0)
    pact_check_status()
    assert not host(dA).any() and not host(dB).any()


def _parity(x, dy, p, what):
    xq = pact_quant_nvfp4(bf16(x))
    dA, dB = pact_lora_adapter_grad(xq, bf16(dy), bf16(p.A), bf16(p.B), p.scale)
    pact_check_status()
    dA_ref, dB_ref = orc.lora_adapter_grad(orc.quantize(x), dy, p.A, p.B, p.alpha)
    for name, got, ref in (("dA", host(dA), dA_ref), ("dB", host(dB), dB_ref)):
        assert_close(got, ref, f"{what} {name}")
        e = _rel_rms(got, ref)
        assert e <= REL_RMS_BOUND, f"{what} {name}: relative RMS error {e:.3g}"


def test_adapter_grad_tiny_workload():
    d = wl.tiny()
    _parity(d["x"], d["dy"], d["proj"], "tiny")


@pytest.mark.parametrize("M,N,K,r", [(1, 64, 64, 4), (333, 192, 448, 12), (1000, 2048, 512, 64),
                                     (257, 384, 1536, 33), (300, 1600, 256, 16)])
def test_adapter_grad_odd_shapes(M, N, K, r):
    rng = np.random.default_rng(M + 7 * N + K + r)
    x = wl.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    p = wl.make_proj(rng, "p", K, N, r, 2.0 * r, w_std=0.05)
    dy = wl.bf16_round(rng.standard_normal((M, N)).astype(np.float32) * 0.1)
    _parity(x, dy, p, "odd")


def test_adapter_grad_q3b_full_size():
    """Query projection of the 3B model at M = 4096, every element compared."""
    d = wl.q3b()
    _parity(d["x"], d["dy"], d["proj"], "q3b")


def test_adapter_grad_mlp3b_gate_up_and_down_full_size():
    """The fused gate|up (K = 3072, N = 16384, r = 32) and down (K = 8192, N = 3072)
    projections of the 3B MLP at M = 4096.  Their output gradients come from the
    out-of-scope parts of the backward, so they are seeded N(0, 1e-2^2) tensors; the
    down projection's input stands in for the SiLU-multiply output."""
    d = wl.mlp3b()
    rng = wl.rng_for(3, salt=77)
    gu = d["gate_up"]
    dgu = wl.bf16_round(wl.normal(rng, (d["x"].shape[0], gu.d_out), 1e-2))
    _parity(d["x"], dgu, gu, "gate_up")
    dn = d["down"]
    h = wl.bf16_round(wl.normal(rng, (d["x"].shape[0], dn.d_in), 0.3))
    _parity(h, d["dy"], dn, "down")
