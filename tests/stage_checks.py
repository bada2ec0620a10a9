"""Per-stage parity helpers: every stage of a GPU chain is checked against the
oracle fed with the GPU's own upstream tensors (read back from the device), so
each stage is held to its per-op bar however many stages precede it: NVFP4
outputs, scales, g and the RMSNorm statistic bit-exact, GEMM and backward outputs
within |gpu - ref| <= 8e-3 |ref| + 2e-3 rms(ref) on the rows compared.  Test
infrastructure: no method arithmetic lives here, only reading back and calling
the oracle."""
import numpy as np
import torch

import oracle as orc

from gpu_helpers import assert_close, assert_nvfp4_equal, host


def q_from_gpu(t) -> "orc.Q":
    """A device NVFP4 tensor as the oracle's Q (codes, logical scales, g)."""
    torch.cuda.synchronize()
    codes = t.codes.cpu().numpy()
    sf = orc.unswizzle_scales(t.sf.cpu().numpy(), t.rows, t.cols // 16)
    return orc.Q(codes=codes, scales=np.ascontiguousarray(sf), g=np.float32(t.g.item()),
                 rows=t.rows, cols=t.cols)


def sample_rows(m: int, n: int = 512, seed: int = 0) -> np.ndarray:
    """All rows when m <= n; else n seeded rows including the first and last rows
    and both sides of every 128-row tile edge among the first and last tiles."""
    if m <= n:
        return np.arange(m)
    edges = {0, m - 1, 127, 128, 255, 256, m - 129, m - 128}
    rng = np.random.default_rng(seed)
    rest = rng.choice(m, size=n, replace=False)
    return np.unique(np.concatenate([rest, np.array(sorted(e for e in edges if 0 <= e < m))]))


def check_fwd(name, y_gpu, xq_gpu, proj, pack_fwd, rows, residual=None):
    """Y = Xhat What^T + (alpha/r)(Xhat A)B [+ residual] on the given rows, from the
    GPU's own NVFP4 input (and residual)."""
    ref = orc.lora_linear_fwd(q_from_gpu(xq_gpu), pack_fwd, proj.A, proj.B, proj.alpha,
                              residual=None if residual is None else host(residual), rows=rows)
    return assert_close(host(y_gpu)[rows], ref, f"{name} forward")


def check_dgrad(name, dx_gpu, dyq_gpu, dy_gpu, proj, pack_bwd, rows, dx_prev=None):
    """dX = dYhat W + (alpha/r)(dY B^T) A^T [+ dx_prev] on the given rows, from the GPU's
    own NVFP4 dY and BF16 dY (and previous dX)."""
    ref = orc.lora_linear_dgrad(q_from_gpu(dyq_gpu), host(dy_gpu), pack_bwd, proj.A, proj.B,
                                proj.alpha, dx_prev=None if dx_prev is None else host(dx_prev),
                                rows=rows)
    return assert_close(host(dx_gpu)[rows], ref, f"{name} input gradient")


def check_quant(name, q_gpu, x_gpu, amax=None):
    """NVFP4 of the GPU's BF16 tensor, every byte; with amax (a device scalar the
    producer wrote) the scale comes from it, and it must equal max |x|."""
    x = host(x_gpu)
    if amax is not None:
        a = np.float32(amax.item())
        assert a.tobytes() == np.float32(np.abs(x).max()).tobytes(), f"{name}: producer amax"
    assert_nvfp4_equal(q_gpu, orc.quantize(x), f"{name} NVFP4")


def check_rmsnorm_quant(name, yq_gpu, rstd_gpu, x_gpu, gamma, eps):
    ref_q, ref_rstd = orc.rmsnorm_quant(host(x_gpu), gamma, eps)
    got = host(rstd_gpu)
    assert np.array_equal(got.view(np.uint32), ref_rstd.view(np.uint32)), f"{name}: rstd"
    assert_nvfp4_equal(yq_gpu, ref_q, f"{name} NVFP4")


def check_silu_quant(name, hq, gq, uq, gu_gpu):
    ref = orc.silu_mul_quant(host(gu_gpu))
    for t, r, w in zip((hq, gq, uq), ref, ("h", "gate", "up")):
        assert_nvfp4_equal(t, r, f"{name} {w}")


def check_silu_bwd(name, dgu_gpu, gq_gpu, uq_gpu, dh_gpu, rows, amax=None):
    g, u = q_from_gpu(gq_gpu), q_from_gpu(uq_gpu)
    ref = orc.silu_mul_bwd_from(orc.dequant_rows(g, rows), orc.dequant_rows(u, rows),
                                host(dh_gpu)[rows])
    got = host(dgu_gpu)
    if amax is not None:
        assert np.float32(amax.item()) == np.float32(np.abs(got).max()), f"{name}: amax"
    return assert_close(got[rows], ref, f"{name} SiLU backward")


def check_rmsnorm_bwd(name, dx_gpu, yq_gpu, gamma, rstd_gpu, dy_gpu, rows, dres=None,
                      amax=None):
    yq = q_from_gpu(yq_gpu)
    ref = orc.rmsnorm_bwd_from_y(orc.dequant_rows(yq, rows), gamma, host(rstd_gpu)[rows],
                                 host(dy_gpu)[rows])
    if dres is not None:
        ref = ref + np.asarray(host(dres)[rows], np.float64)
    got = host(dx_gpu)
    if amax is not None:
        assert np.float32(amax.item()) == np.float32(np.abs(got).max()), f"{name}: amax"
    return assert_close(got[rows], ref, f"{name} RMSNorm backward")
