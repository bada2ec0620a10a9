"""Helpers shared by the GPU parity tests: moving seeded inputs to the device and
reading device NVFP4 tensors back for comparison with the oracle.  No method
arithmetic lives here."""
import numpy as np
import torch

import oracle as orc
from nvfp4_frozen_projection_gb300 import NVFP4


def dev():
    return torch.device("cuda", 0)


def bf16(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).to(dev())


def f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev())


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def nvfp4_to_device(q: "orc.Q") -> NVFP4:
    """Upload a seeded, host-constructed NVFP4 tensor (codes, logical scales, g)."""
    t = NVFP4.empty(q.rows, q.cols, dev())
    t.codes.copy_(torch.from_numpy(np.ascontiguousarray(q.codes)))
    t.sf.copy_(torch.from_numpy(orc.swizzle_scales(q.scales)))
    t.g.fill_(float(q.g))
    return t


def assert_nvfp4_equal(gpu: NVFP4, ref: "orc.Q", what=""):
    """Bit-exact comparison: codes, every byte of the swizzled scale array (pads
    included) and g."""
    torch.cuda.synchronize()
    codes = gpu.codes.cpu().numpy()
    sf = gpu.sf.cpu().numpy()
    g = np.float32(gpu.g.cpu().numpy()[0])
    assert g.tobytes() == np.float32(ref.g).tobytes(), f"{what}: g {g!r} != {ref.g!r}"
    want_sf = orc.swizzle_scales(ref.scales)
    bad_sf = np.nonzero(sf != want_sf)[0]
    assert bad_sf.size == 0, f"{what}: {bad_sf.size} scale bytes differ, first at {bad_sf[:5]}"
    bad = np.argwhere(codes != ref.codes)
    assert bad.size == 0, f"{what}: {len(bad)} code bytes differ, first at {bad[:5].tolist()}"


def assert_close(gpu, ref, what="", rms_ref=None):
    ok, worst, idx = orc.check_close(gpu, ref, rms_ref=rms_ref)
    assert ok, f"{what}: outside tolerance, worst |err|/bound = {worst:.3f} at {idx}"
    return worst
