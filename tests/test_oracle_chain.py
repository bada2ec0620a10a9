"""Pins for the oracle chains (oracle/chain.py).  CPU only.

round_bf16 is checked against PyTorch's FP32 -> BF16 conversion (round to nearest
even) on FP32-representable values, ties and subnormals included.

The chains compose per-op oracle functions that are pinned one by one; what is
pinned here is the composition: the wiring of residuals, the order of the
accumulations and which gradient flows where.  Each chain is compared with FP64
autograd through the same layer written without quantisation (a plain forward, no
hand-written backward).  The chains quantise every GEMM operand to NVFP4, so the two
agree only up to the format's error (a few percent per operand); a dropped term,
a wrong sign, a missing residual or a transposed adapter moves the result by far
more than the bounds used below.  A second check zeroes the weights of later
projections so that a residual path has to reproduce its input exactly.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from oracle import chain
from nvfp4_frozen_projection_gb300 import workloads as wl


# ------------------------------------------------------------------ round_bf16
def test_round_bf16_matches_torch_conversion():
    rng = np.random.default_rng(3)
    vals = [rng.standard_normal(20000).astype(np.float32) * np.float32(s)
            for s in (1.0, 1e-3, 1e4, 1e-38, 1e-40, 1e37)]
    # exact ties: a BF16 value plus half an ulp (bit 15 set, lower bits clear)
    base = (rng.integers(0, 2 ** 16, 5000, dtype=np.uint32) << 16) | np.uint32(0x8000)
    ties = base.view(np.float32)
    ties = ties[np.isfinite(ties)]
    x = np.concatenate(vals + [ties, np.array([0.0, -0.0, 1.0, -2.5], np.float32)])
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = chain.round_bf16(x.astype(np.float64))
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(want[finite]))


# ------------------------------------------------------ unquantised FP64 layer
def _t(a):
    return torch.tensor(np.asarray(a, np.float64))


def _lin(x, p):
    W, A, B = _t(p.W), _t(p.A), _t(p.B)
    return x @ W.T + (p.alpha / A.shape[1]) * ((x @ A) @ B)


def _rms(x, gamma, eps):
    return x * torch.rsqrt((x * x).mean(dim=1, keepdim=True) + float(eps)) * _t(gamma)


def _silu_mul(gu):
    I = gu.shape[1] // 2
    g, u = gu[:, :I], gu[:, I:]
    return g * torch.sigmoid(g) * u


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _small_layer():
    return wl.layer3b(m=48, hidden=128, kv=64, inter=256)


def _layer_errors(d):
    """Relative errors of the oracle chain against FP64 autograd of the unquantised
    layer: forward activations and the two input gradients."""
    o = chain.decoder_layer(d)
    x = _t(d["x"]).requires_grad_()
    attn = _t(d["attn"]).requires_grad_()
    n1 = _rms(x, d["gamma1"], d["eps"])
    q, k, v = (_lin(n1, d[n]) for n in ("q", "k", "v"))
    h1 = _lin(attn, d["o"]) + x
    gu = _lin(_rms(h1, d["gamma2"], d["eps"]), d["gate_up"])
    out = _lin(_silu_mul(gu), d["down"]) + h1
    loss = ((out * _t(d["dy"])).sum() + (q * _t(d["dq"])).sum() + (k * _t(d["dk"])).sum()
            + (v * _t(d["dv"])).sum())
    dx, dattn = torch.autograd.grad(loss, (x, attn))
    got = {n: o[n] for n in ("q", "k", "v", "h1", "gu", "out")}
    err = {n: _rel(got[n], ref.detach())
           for n, ref in (("q", q), ("k", k), ("v", v), ("h1", h1), ("gu", gu), ("out", out))}
    err["dattn"] = _rel(o["dattn"], dattn)
    err["dx"] = _rel(o["dx"], dx)
    return err


# Bounds: the chain's own NVFP4 error measured 0.06-0.12 (forward) and 0.06-0.08
# (gradients) at this size; every planted mistake below moves at least one of
# these quantities past them.
FWD_BOUND = 0.2
GRAD_BOUND = 0.15


def _within(err):
    return (all(err[n] < FWD_BOUND for n in ("q", "k", "v", "h1", "gu", "out"))
            and err["dattn"] < GRAD_BOUND and err["dx"] < GRAD_BOUND)


def test_decoder_layer_against_fp64_autograd():
    err = _layer_errors(_small_layer())
    assert _within(err), err


_FWD, _DGRAD = chain.lora_linear_fwd, chain.lora_linear_dgrad
_RMS_BWD, _SILU_BWD = chain.rmsnorm_bwd, chain.silu_mul_bwd


def _silu_bwd_swapped(gq, uq, dh):
    r = _SILU_BWD(gq, uq, dh)
    i = r.shape[1] // 2
    return np.concatenate([r[:, i:], r[:, :i]], axis=1)


def _fwd_without_base(xq, w, A, B, alpha, residual=None):
    zero_w = orc.quantize(np.zeros((w.rows, w.cols), np.float32))
    return _FWD(xq, zero_w, A, B, alpha, residual)


PLANTED = {
    "LoRA sign": ("lora_linear_fwd", lambda xq, w, A, B, al, residual=None:
                  _FWD(xq, w, A, -np.asarray(B), al, residual)),
    "residual dropped": ("lora_linear_fwd", lambda xq, w, A, B, al, residual=None:
                         _FWD(xq, w, A, B, al, None)),
    "frozen GEMM dropped": ("lora_linear_fwd", _fwd_without_base),
    "scale alpha instead of alpha/r": ("lora_linear_fwd", lambda xq, w, A, B, al, residual=None:
                                       _FWD(xq, w, A, B, al * np.asarray(A).shape[1], residual)),
    "dgrad LoRA sign": ("lora_linear_dgrad", lambda q, dy, w, A, B, al, dx_prev=None:
                        _DGRAD(q, dy, w, -np.asarray(A), B, al, dx_prev)),
    "dgrad frozen GEMM dropped": ("lora_linear_dgrad", lambda q, dy, w, A, B, al, dx_prev=None:
                                  _DGRAD(orc.quantize(np.zeros((q.rows, q.cols), np.float32)),
                                         dy, w, A, B, al, dx_prev)),
    "q, k and v gradients not accumulated": ("lora_linear_dgrad",
                                            lambda q, dy, w, A, B, al, dx_prev=None:
                                            _DGRAD(q, dy, w, A, B, al)),
    "RMSNorm residual gradient dropped": ("rmsnorm_bwd", lambda yq, g, r, dy, dres=None:
                                          _RMS_BWD(yq, g, r, dy)),
    "SiLU gradients swapped": ("silu_mul_bwd", _silu_bwd_swapped),
}


@pytest.mark.parametrize("mistake", sorted(PLANTED))
def test_planted_mistake_is_caught(mistake, monkeypatch):
    """A mistake planted in the oracle chain (on the CPU) breaks the autograd pin."""
    name, fn = PLANTED[mistake]
    monkeypatch.setattr(chain, name, fn)
    assert not _within(_layer_errors(_small_layer()))


def test_mlp_against_fp64_autograd():
    d = wl.mlp3b(m=40, hidden=128, inter=256)
    o = chain.mlp(d["x"], d["gate_up"], d["down"], d["dy"])
    x = _t(d["x"]).requires_grad_()
    gu = _lin(x, d["gate_up"])
    out = _lin(_silu_mul(gu), d["down"])
    (dx,) = torch.autograd.grad((out * _t(d["dy"])).sum(), (x,))
    # the MLP input is not normalised, so the NVFP4 error is larger here (0.10 /
    # 0.18 / 0.15 measured)
    assert _rel(o["gu"], gu.detach()) < 0.15
    assert _rel(o["out"], out.detach()) < 0.25
    assert _rel(o["dx"], dx) < 0.22


def test_attention_inputs_against_fp64_autograd():
    d = wl.attn1b(m=40, hidden=128, kv=64)
    o = chain.attention_inputs(d["x"], d["gamma"], d["projs"], d["dys"], d["eps"])
    x = _t(d["x"]).requires_grad_()
    n = _rms(x, d["gamma"], d["eps"])
    ys = [_lin(n, p) for p in d["projs"]]
    loss = sum((y * _t(dy)).sum() for y, dy in zip(ys, d["dys"]))
    (dx,) = torch.autograd.grad(loss, (x,))
    for got, ref in zip(o["y"], ys):
        assert _rel(got, ref.detach()) < FWD_BOUND
    assert _rel(o["dx"], dx) < GRAD_BOUND


def test_decoder_layer_residual_paths_are_exact():
    """With o, gate|up and down zeroed (weights and adapters), h1 = x and out = h1
    exactly, and the input gradient reduces to dy pushed through the two residuals
    plus the q/k/v gradients through the first RMSNorm."""
    d = _small_layer()
    for n in ("o", "gate_up", "down"):
        p = d[n]
        p.W = np.zeros_like(p.W)
        p.B = np.zeros_like(p.B)
    o = chain.decoder_layer(d)
    assert np.array_equal(o["h1"], d["x"])
    assert np.array_equal(o["out"], d["x"])
    assert not np.any(o["dattn"])
    assert not np.any(o["dxn2"])
    # dh1 = dy (RMSNorm-2 backward sees a zero incoming gradient, plus dres = dy)
    assert np.array_equal(o["dh1"], d["dy"])
    # dx = RMSNorm-1 backward of the q/k/v gradient + dh1
    want = chain.round_bf16(orc.rmsnorm_bwd(o["xq1"], d["gamma1"], o["rstd1"], o["dxn1"],
                                            dres=d["dy"]))
    assert np.array_equal(o["dx"], want)
    # and without the q/k/v gradients dx is dy itself
    d["dq"] = np.zeros_like(d["dq"])
    d["dk"] = np.zeros_like(d["dk"])
    d["dv"] = np.zeros_like(d["dv"])
    o = chain.decoder_layer(d)
    assert np.array_equal(o["dx"], d["dy"])
