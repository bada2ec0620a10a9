"""Library calls queued behind other work on their stream.  These tests queue each
two-pass call (its amax or statistic kernel, then the encode that reads the amax)
behind a copy, a weight pack and the call itself, without synchronising, and
require the oracle's bytes every time: an encode that read the amax before its
producer finished (any overlap of consecutive kernels that did not wait for the
previous one) gives a different per-tensor scale."""
import numpy as np
import pytest
import torch

import oracle as orc
import nvfp4_frozen_projection_gb300 as pk
from nvfp4_frozen_projection_gb300 import workloads as wl

from gpu_helpers import assert_nvfp4_equal, bf16, f32

pytestmark = pytest.mark.gpu

M, H = 4096, 3072


@pytest.fixture(scope="module")
def inputs():
    rng = np.random.default_rng(31)
    x = wl.bf16_round((rng.standard_t(3, (M, H)) / np.sqrt(3.0)).astype(np.float32))
    gamma = wl.bf16_round((1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    W = (rng.standard_normal((1024, H)) * 0.02).astype(np.float32)
    return x, gamma, W


def _before(kind, xd, gd, wd):
    """Work queued ahead of the call on the same stream (not waited for)."""
    if kind == "copy":
        xd.clone()
    elif kind == "pack":
        pk.pact_pack_weight_fwd(wd)
    elif kind == "quant":
        pk.pact_quant_nvfp4(xd)
    elif kind == "rmsnorm":
        pk.pact_rmsnorm_quant(xd, gd)


@pytest.mark.parametrize("kind", ["copy", "pack", "quant", "rmsnorm"])
def test_rmsnorm_quant_behind_queued_work(inputs, kind):
    x, gamma, W = inputs
    ref, rstd_ref = orc.rmsnorm_quant(x, gamma)
    xd, gd, wd = bf16(x), bf16(gamma), f32(W)
    yq, rstd = pk.pact_rmsnorm_quant(xd, gd)
    for it in range(6):
        _before(kind, xd, gd, wd)
        pk.pact_rmsnorm_quant(xd, gd, out=yq, rstd=rstd)
        assert_nvfp4_equal(yq, ref, f"RMSNorm -> NVFP4 behind {kind}, round {it}")
    pk.pact_check_status()


@pytest.mark.parametrize("kind", ["copy", "pack", "rmsnorm"])
def test_quant_behind_queued_work(inputs, kind):
    x, gamma, W = inputs
    ref = orc.quantize(x)
    xd, gd, wd = bf16(x), bf16(gamma), f32(W)
    q = pk.pact_quant_nvfp4(xd)
    for it in range(6):
        _before(kind, xd, gd, wd)
        pk.pact_quant_nvfp4(xd, out=q)
        assert_nvfp4_equal(q, ref, f"quant behind {kind}, round {it}")
    pk.pact_check_status()
