"""GPU parity: NVFP4 quantisation, weight packs and the exp recipe must match the
oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle as orc
from nvfp4_frozen_projection_gb300 import (pact_pack_weight_bwd, pact_pack_weight_fwd,
                                           pact_quant_nvfp4, pact_test_pexp, pact_check_status)
from nvfp4_frozen_projection_gb300 import workloads as wl

from gpu_helpers import assert_nvfp4_equal, bf16, f32, host

pytestmark = pytest.mark.gpu


def _quant_case(x):
    xb = bf16(x)
    q = pact_quant_nvfp4(xb)
    pact_check_status()
    ref = orc.quantize(host(xb))
    assert_nvfp4_equal(q, ref, f"quant {x.shape}")


@pytest.mark.parametrize("shape", [(64, 256), (1, 64), (127, 192), (300, 1088), (129, 3072)])
def test_quant_random_shapes(shape):
    rng = np.random.default_rng(sum(shape))
    x = rng.standard_normal(shape).astype(np.float32) * np.exp(rng.uniform(-4, 4, (shape[0], 1)))
    _quant_case(x.astype(np.float32))


def test_quant_edge_values():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((130, 128)).astype(np.float32)
    x[0, :16] = 0.0                         # zero block
    x[1, :] = -0.0                          # negative zeros
    x[2, 5] = 1e4                           # tensor max, far above the rest
    x[3, :16] = 1e-3                        # constant block
    x[4, :16] = 3e-38                       # tiny block (E4M3 underflow to 0)
    x[5, 16:32] = -x[5, 16:32]
    _quant_case(x)


def test_quant_zero_tensor():
    _quant_case(np.zeros((64, 64), np.float32))


def test_quant_strided_rows_and_amax():
    rng = np.random.default_rng(8)
    full = rng.standard_normal((96, 512)).astype(np.float32)
    xb = bf16(full)
    view = xb[:, 128:384]                  # row stride 512, 256 columns
    amax = torch.tensor([float(np.abs(host(view)).max())], dtype=torch.float32, device=xb.device)
    q1 = pact_quant_nvfp4(view)
    q2 = pact_quant_nvfp4(view, amax=amax)
    ref = orc.quantize(host(view))
    assert_nvfp4_equal(q1, ref, "strided")
    assert_nvfp4_equal(q2, ref, "strided + amax")


def test_quant_workloads_full_size():
    """Workload 2's X (outlier channels) and dY at full size, every byte."""
    d = wl.q3b()
    _quant_case(d["x"])
    _quant_case(d["dy"])


def test_quant_tiny_workload():
    d = wl.tiny()
    _quant_case(d["x"])
    _quant_case(d["dy"])


@pytest.mark.parametrize("NK", [(64, 64), (256, 256), (192, 320), (3072, 3072)])
def test_weight_packs_bit_exact(NK):
    N, K = NK
    rng = np.random.default_rng(N + K)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    W[rng.integers(0, N), rng.integers(0, K)] = 0.7
    Wd = f32(W)
    fwd = pact_pack_weight_fwd(Wd)
    bwd = pact_pack_weight_bwd(Wd)
    pact_check_status()
    rf, rb = orc.pack_weight(W)
    assert_nvfp4_equal(fwd, rf, "pack fwd")
    assert_nvfp4_equal(bwd, rb, "pack bwd")


def test_pexp_bit_exact():
    xs = np.concatenate([
        np.linspace(-110, 92, 400001, dtype=np.float32),
        np.float32([0.0, -0.0, 88.72283172607422, 88.72283935546875, -103.97207, -103.9721,
                    1e-30, -1e-30, 0.34657359, -0.34657359, np.inf, -np.inf]),
        (np.random.default_rng(9).standard_normal(100000) * 20).astype(np.float32),
    ])
    y = pact_test_pexp(f32(xs)).cpu().numpy()
    want = orc.pexp(xs)
    assert y.tobytes() == want.tobytes() or np.array_equal(
        y.view(np.uint32), want.view(np.uint32)), \
        f"{np.count_nonzero(y.view(np.uint32) != want.view(np.uint32))} values differ"
