"""The no-allocation LoRA linear forward.

Some callers cannot allocate device memory or pass a workspace (a plugin that is
handed only inputs and outputs, code running during CUDA graph capture, a runtime
with a fixed memory budget).  pact_lora_linear_fwd_noalloc serves them with a
fixed scratch array inside the library.  This test calls it through the C ABI
twice in a row, with different shapes and data, and checks each result against
the regular entry point (which takes a workspace) within the parity tolerance.
It also checks that a call needing more scratch than the fixed array is refused
without launching.  The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import nvfp4_frozen_projection_gb300 as pk
from nvfp4_frozen_projection_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _case(seed, M, N, K, r):
    rng = np.random.default_rng(seed)
    x = wl.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    p = wl.make_proj(rng, "p", K, N, r, 2.0 * r, w_std=0.05)
    dev = torch.device("cuda", 0)
    xq = pk.pact_quant_nvfp4(torch.from_numpy(x).to(dev).bfloat16())
    wf = pk.pact_pack_weight_fwd(torch.from_numpy(p.W).to(dev))
    A = torch.from_numpy(p.A).to(dev).bfloat16()
    B = torch.from_numpy(p.B).to(dev).bfloat16()
    return xq, wf, A, B, p.scale


def test_noalloc_matches_regular_entry_point_twice():
    cases = [(1, 256, 512, 256, 16), (2, 200, 384, 640, 8)]
    for seed, M, N, K, r in cases:
        xq, wf, A, B, scale = _case(seed, M, N, K, r)
        y_ref = pk.pact_lora_linear_fwd(xq, wf, A, B, scale)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        pk.pact_lora_linear_fwd_noalloc(xq, wf, A, B, scale, y)
        pk.pact_check_status()
        got, ref = y.float().cpu().numpy(), y_ref.float().cpu().numpy()
        ok, worst, idx = orc.check_close(got, ref)
        assert ok, f"case {seed}: worst |err|/bound {worst:.3f} at {idx}"


def test_noalloc_rejects_oversized_calls():
    lib = pk.load_library()
    cap = int(lib.pact_lora_linear_fwd_noalloc_max_scratch())
    assert cap == 16 << 20
    # scratch: align256(4 M rp) + align256(2 N rp) + align256(2 K rp), rp = 16: > 16 MiB
    M, N, K, r = 262144, 64, 64, 16
    assert lib.pact_lora_linear_fwd_workspace_size(M, N, K, r) > cap
    xq = pk.NVFP4.empty(1, 64)        # small real buffers; the shape fields claim more
    wf = pk.NVFP4.empty(N, K)
    xq.rows, xq.cols = M, K
    A = torch.zeros((K, r), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((r, N), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pk.PactError) as ei:
        pk.pact_lora_linear_fwd_noalloc(xq, wf, A, B, 1.0, y)
    assert ei.value.code == 2 and "scratch" in str(ei.value)
    torch.cuda.synchronize()
