"""Out-of-bounds evidence for every entry point: each output buffer, and the
workspace, is followed by guard bytes of a fixed pattern and checked after the
call; the outputs themselves start as garbage, so that a byte the call should
write but leaves alone shows up in the parity comparisons that follow.  Shapes are
ragged (rows not a multiple of 128, column counts off the tile widths, ranks off
the padded widths), so the padding logic of every kernel is exercised."""
import numpy as np
import pytest
import torch

import oracle as orc
import nvfp4_frozen_projection_gb300 as pk
from nvfp4_frozen_projection_gb300 import NVFP4
from nvfp4_frozen_projection_gb300 import workloads as wl

from gpu_helpers import assert_close, assert_nvfp4_equal, bf16, f32, host

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class _Guarded:
    """nbytes of device memory (filled with garbage) followed by GUARD pattern bytes."""

    def __init__(self, nbytes, dtype=torch.uint8, shape=None):
        nbytes = int(nbytes)
        self.n = nbytes
        self.buf = torch.full((nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        g = torch.Generator(device="cuda")
        g.manual_seed(nbytes)
        self.buf[:nbytes] = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda",
                                          generator=g)
        t = self.buf[:nbytes].view(dtype)
        self.t = t.view(shape) if shape is not None else t

    def intact(self):
        torch.cuda.synchronize()
        tail = self.buf[self.n:].cpu().numpy()
        return bool(np.all(tail == PATTERN))


_ALL = []


def _g(nbytes, dtype=torch.uint8, shape=None):
    x = _Guarded(nbytes, dtype, shape)
    _ALL.append(x)
    return x.t


def _nv(rows, cols):
    sf = ((rows + 127) // 128 * 128) * ((cols // 16 + 3) // 4 * 4)
    return NVFP4(_g(rows * cols // 2, shape=(rows, cols // 2)), _g(sf), _g(4, torch.float32), rows,
                 cols)


def _bf(rows, cols):
    return _g(rows * cols * 2, torch.bfloat16, (rows, cols))


@pytest.fixture(autouse=True)
def guarded_workspace(monkeypatch):
    """Every call's workspace is exactly the size the library asks for, guarded."""
    _ALL.clear()

    def ws(nbytes, device):
        return _g(max(256, int(nbytes)))
    monkeypatch.setattr(pk, "_workspace", ws)
    yield
    bad = [i for i, x in enumerate(_ALL) if not x.intact()]
    assert not bad, f"guard bytes overwritten after buffers {bad}"


def _data(seed, shape, std=1.0):
    rng = np.random.default_rng(seed)
    return wl.bf16_round((rng.standard_normal(shape) * std).astype(np.float32))


M, N, K, R = 200, 192, 320, 12   # ragged rows, 192 = 1.5 tiles of 128, rank padded to 16


def _proj(seed, n_out, k_in, r):
    return wl.make_proj(np.random.default_rng(seed), "p", k_in, n_out, r, 2.0 * r, w_std=0.05)


def _gate_up_perm(I):
    """Row order of the gate|up forward pack: gate and up rows interleaved in groups of 32."""
    return np.concatenate([np.r_[32 * j:32 * j + 32, I + 32 * j:I + 32 * j + 32]
                           for j in range(I // 32)])


# one test per entry point of the library --------------------------------------------

def test_quant_nvfp4():
    x = _data(1, (M, K))
    q = pk.pact_quant_nvfp4(bf16(x), out=_nv(M, K))
    assert_nvfp4_equal(q, orc.quantize(x), "quant")
    wide = _bf(M, K + 64)           # row stride above K: the tail of each row is not read
    wide[:, :K].copy_(bf16(x))
    q2 = pk.pact_quant_nvfp4(wide[:, :K], out=_nv(M, K))
    assert_nvfp4_equal(q2, orc.quantize(x), "quant, strided rows")
    pk.pact_check_status()


def test_pack_weight_fwd():
    W = (np.random.default_rng(2).standard_normal((N, K)) * 0.05).astype(np.float32)
    assert_nvfp4_equal(pk.pact_pack_weight_fwd(f32(W), out=_nv(N, K)), orc.pack_weight(W)[0],
                       "pack fwd")
    pk.pact_check_status()


def test_pack_weight_bwd():
    W = (np.random.default_rng(2).standard_normal((N, K)) * 0.05).astype(np.float32)
    assert_nvfp4_equal(pk.pact_pack_weight_bwd(f32(W), out=_nv(K, N)), orc.pack_weight(W)[1],
                       "pack bwd")
    pk.pact_check_status()


def test_pack_weight_fwd_gate_up():
    W = (np.random.default_rng(3).standard_normal((2 * N, K)) * 0.05).astype(np.float32)
    q = pk.pact_pack_weight_fwd_gate_up(f32(W), out=_nv(2 * N, K))
    assert_nvfp4_equal(q, orc.pack_weight(W[_gate_up_perm(N)])[0], "pack fwd gate|up")
    pk.pact_check_status()


def test_lora_linear_fwd():
    p = _proj(4, N, K, R)
    x, res = _data(5, (M, K)), _data(6, (M, N))
    xq = pk.pact_quant_nvfp4(bf16(x))
    amax = _g(4, torch.float32)
    y = pk.pact_lora_linear_fwd(xq, pk.pact_pack_weight_fwd(f32(p.W)), bf16(p.A), bf16(p.B),
                                p.scale, residual=bf16(res), y=_bf(M, N), out_amax=amax)
    want = orc.lora_linear_fwd(orc.quantize(x), orc.pack_weight(p.W)[0], p.A, p.B, p.alpha,
                               residual=res)
    assert_close(host(y), want, "forward")
    assert amax.item() == np.abs(host(y)).max()
    pk.pact_check_status()


def test_lora_linear_fwd_noalloc():
    p = _proj(4, N, K, R)
    xq = pk.pact_quant_nvfp4(bf16(_data(5, (M, K))))
    wf = pk.pact_pack_weight_fwd(f32(p.W))
    y = pk.pact_lora_linear_fwd_noalloc(xq, wf, bf16(p.A), bf16(p.B), p.scale, _bf(M, N))
    ref = pk.pact_lora_linear_fwd(xq, wf, bf16(p.A), bf16(p.B), p.scale)
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    pk.pact_check_status()


def test_lora_linear_fwd_gate_up():
    pg = _proj(7, 2 * N, K, R)
    xq = pk.pact_quant_nvfp4(bf16(_data(5, (M, K))))
    yg, a3 = pk.pact_lora_linear_fwd_gate_up(xq, pk.pact_pack_weight_fwd_gate_up(f32(pg.W)),
                                             bf16(pg.A), bf16(pg.B), pg.scale,
                                             y=_bf(M, 2 * N), amax3=_g(12, torch.float32))
    ref = pk.pact_lora_linear_fwd(xq, pk.pact_pack_weight_fwd(f32(pg.W)), bf16(pg.A),
                                  bf16(pg.B), pg.scale)
    assert torch.equal(yg.view(torch.int16), ref.view(torch.int16))
    gu = host(yg)
    want = np.float32([np.abs(orc.silu_mul_fp32(gu)).max(), np.abs(gu[:, :N]).max(),
                       np.abs(gu[:, N:]).max()])
    assert a3.cpu().numpy().view(np.uint32).tolist() == want.view(np.uint32).tolist()
    pk.pact_check_status()


def test_lora_linear_dgrad():
    p = _proj(8, N, K, R)
    dy = _data(9, (M, N), 0.1)
    wb = pk.pact_pack_weight_bwd(f32(p.W))
    dyq = pk.pact_quant_nvfp4(bf16(dy))
    dx = pk.pact_lora_linear_dgrad(dyq, bf16(dy), wb, bf16(p.A), bf16(p.B), p.scale,
                                   dx=_bf(M, K))
    owb = orc.pack_weight(p.W)[1]
    assert_close(host(dx), orc.lora_linear_dgrad(orc.quantize(dy), dy, owb, p.A, p.B, p.alpha),
                 "dgrad")
    dx2 = _bf(M, K)
    dx2.copy_(dx)
    pk.pact_lora_linear_dgrad(dyq, bf16(dy), wb, bf16(p.A), bf16(p.B), p.scale, dx=dx2,
                              accumulate=True)
    assert_close(host(dx2), orc.lora_linear_dgrad(orc.quantize(dy), dy, owb, p.A, p.B, p.alpha,
                                                  dx_prev=host(dx)), "dgrad accumulate")
    pk.pact_check_status()


def test_lora_linear_dgrad_q():
    p = _proj(8, N, K, R)
    dy = _data(9, (M, N), 0.1)
    wb = pk.pact_pack_weight_bwd(f32(p.W))
    dx, dyq = pk.pact_lora_linear_dgrad_q(bf16(dy), wb, bf16(p.A), bf16(p.B), p.scale,
                                          dyq=_nv(M, N), dx=_bf(M, K))
    assert_nvfp4_equal(dyq, orc.quantize(dy), "fused dY")
    ref = pk.pact_lora_linear_dgrad(pk.pact_quant_nvfp4(bf16(dy)), bf16(dy), wb, bf16(p.A),
                                    bf16(p.B), p.scale)
    assert torch.equal(dx.view(torch.int16), ref.view(torch.int16))
    pk.pact_check_status()


def test_lora_adapter_grad():
    p = _proj(8, N, K, R)
    x, dy = _data(10, (M, K)), _data(9, (M, N), 0.1)
    dA, dB = pk.pact_lora_adapter_grad(pk.pact_quant_nvfp4(bf16(x)), bf16(dy), bf16(p.A),
                                       bf16(p.B), p.scale,
                                       dA=_g(K * R * 4, torch.float32, (K, R)),
                                       dB=_g(R * N * 4, torch.float32, (R, N)))
    rA, rB = orc.lora_adapter_grad(orc.quantize(x), dy, p.A, p.B, p.alpha)
    assert_close(host(dA), rA, "dA")
    assert_close(host(dB), rB, "dB")
    pk.pact_check_status()


def _norm_inputs(H):
    x = _data(11, (M, H))
    gamma = wl.bf16_round(1.0 + 0.1 * np.random.default_rng(12).standard_normal(H)
                          .astype(np.float32))
    return x, gamma


def test_rmsnorm_quant():
    x, gamma = _norm_inputs(K)
    yq, rstd = pk.pact_rmsnorm_quant(bf16(x), bf16(gamma), 1e-5, out=_nv(M, K),
                                     rstd=_g(M * 4, torch.float32))
    rq, rr = orc.rmsnorm_quant(x, gamma)
    assert_nvfp4_equal(yq, rq, "rmsnorm")
    assert np.array_equal(host(rstd).view(np.uint32), rr.view(np.uint32))
    pk.pact_check_status()


def test_rmsnorm_bwd():
    x, gamma = _norm_inputs(K)
    yq, rstd = pk.pact_rmsnorm_quant(bf16(x), bf16(gamma), 1e-5)
    rq, rr = orc.rmsnorm_quant(x, gamma)
    dy = _data(13, (M, K), 0.1)
    amax = _g(4, torch.float32)
    dx = pk.pact_rmsnorm_bwd(yq, bf16(gamma), rstd, bf16(dy), dres=bf16(dy), dx=_bf(M, K),
                             out_amax=amax)
    assert_close(host(dx), orc.rmsnorm_bwd(rq, gamma, rr, dy, dres=dy), "rmsnorm bwd")
    assert amax.item() == np.abs(host(dx)).max()
    pk.pact_check_status()


def test_silu_mul_quant():
    gu = _data(14, (M, 2 * N))
    hq, gq, uq = pk.pact_silu_mul_quant(bf16(gu), outs=(_nv(M, N), _nv(M, N), _nv(M, N)))
    for t, r_, w in zip((hq, gq, uq), orc.silu_mul_quant(gu), ("h", "gate", "up")):
        assert_nvfp4_equal(t, r_, f"silu {w}")
    pk.pact_check_status()


def test_silu_mul_bwd():
    gu, dh = _data(14, (M, 2 * N)), _data(15, (M, N), 0.1)
    _, gq, uq = pk.pact_silu_mul_quant(bf16(gu))
    amax = _g(4, torch.float32)
    dgu = pk.pact_silu_mul_bwd(gq, uq, bf16(dh), dgateup=_bf(M, 2 * N), out_amax=amax)
    _, rg, ru = orc.silu_mul_quant(gu)
    assert_close(host(dgu), orc.silu_mul_bwd(rg, ru, dh), "silu bwd")
    assert amax.item() == np.abs(host(dgu)).max()
    pk.pact_check_status()
