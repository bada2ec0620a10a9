"""CPU oracle for the NVFP4 LoRA-linear hot path.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code with
the CUDA library and never calls it.

Source: "PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs".
  * Table 6: NVFP4 = E2M1 elements, one E4M3 scale per block of 16, 4.5 bits/elt.
  * Table 7: frozen projections are NVFP4 GEMMs with FP32 accumulation and BF16
    output; cached forward and backward NVFP4 weight layouts; RMSNorm keeps its
    NVFP4 output and an FP32 per-token statistic; SiLU-multiply keeps separate
    NVFP4 gate/up copies; the LoRA branch runs BF16 GEMMs on the reconstructed
    (dequantised) shared input.
  * Abstract: frozen projections run as native NVFP4 GEMMs; forward nonlinear ops
    read BF16 inputs.

The steps whose FP32 operation order decides a bit (encodings, RMSNorm statistic,
SiLU) are plain C (``nvfp4_oracle.c``); contractions and backward ops are FP64
numpy on exactly dequantised operands.  Every function has a "pin" test in
tests/ that checks it against something other than itself.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from .build import build_oracle

_LIB = None

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i64 = ctypes.c_int64


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(build_oracle())
        sig = {
            "orc_e2m1_decode": (ctypes.c_float, [ctypes.c_uint32]),
            "orc_e4m3_decode": (ctypes.c_float, [ctypes.c_uint32]),
            "orc_e2m1_encode": (ctypes.c_uint32, [ctypes.c_float]),
            "orc_e4m3_encode": (ctypes.c_uint32, [ctypes.c_float]),
            "orc_amax": (ctypes.c_float, [_f32p, _i64]),
            "orc_global_scale": (ctypes.c_float, [ctypes.c_float]),
            "orc_quant_rows": (None, [_f32p, _i64, _i64, _i64, ctypes.c_float, _u8p, _u8p]),
            "orc_pack_weight": (None, [_f32p, _i64, _i64, ctypes.c_float, _u8p, _u8p, _u8p, _u8p]),
            "orc_dequant_rows": (None, [_u8p, _u8p, ctypes.c_float, _i64, _i64, _f64p]),
            "orc_rmsnorm_rows": (None, [_f32p, _f32p, _i64, _i64, ctypes.c_float, _f32p, _f32p]),
            "orc_pexp": (ctypes.c_float, [ctypes.c_float]),
            "orc_pexp_array": (None, [_f32p, _i64, _f32p]),
            "orc_silu_mul_rows": (None, [_f32p, _i64, _i64, _f32p]),
            "orc_e2m1_encode_array": (None, [_f32p, _i64, _u8p]),
            "orc_e4m3_encode_array": (None, [_f32p, _i64, _u8p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _p(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


# --------------------------------------------------------------------- codecs
def e2m1_decode(code: int) -> float:
    return float(_lib().orc_e2m1_decode(int(code)))


def e4m3_decode(byte: int) -> float:
    return float(_lib().orc_e4m3_decode(int(byte)))


def e2m1_encode(v: float) -> int:
    return int(_lib().orc_e2m1_encode(float(np.float32(v))))


def e4m3_encode(v: float) -> int:
    return int(_lib().orc_e4m3_encode(float(np.float32(v))))


def e2m1_encode_array(v) -> np.ndarray:
    v = _f32(v).ravel()
    out = np.empty(v.size, np.uint8)
    _lib().orc_e2m1_encode_array(_p(v, ctypes.c_float), v.size, _p(out, ctypes.c_uint8))
    return out


def e4m3_encode_array(v) -> np.ndarray:
    v = _f32(v).ravel()
    out = np.empty(v.size, np.uint8)
    _lib().orc_e4m3_encode_array(_p(v, ctypes.c_float), v.size, _p(out, ctypes.c_uint8))
    return out


E2M1_TABLE = None
E4M3_TABLE = None


def _tables():
    global E2M1_TABLE, E4M3_TABLE
    if E2M1_TABLE is None:
        E2M1_TABLE = np.array([e2m1_decode(c) for c in range(16)], np.float64)
        E4M3_TABLE = np.array([e4m3_decode(b) for b in range(256)], np.float64)
    return E2M1_TABLE, E4M3_TABLE


# --------------------------------------------------------------- NVFP4 tensor
@dataclass
class Q:
    """An NVFP4 tensor [rows, cols]: codes [rows, cols/2] (even column in the low
    nibble), logical E4M3 block scales [rows, cols/16] and the FP32 per-tensor g."""
    codes: np.ndarray
    scales: np.ndarray
    g: np.float32
    rows: int
    cols: int


def amax(x) -> np.float32:
    x = _f32(x).ravel()
    return np.float32(_lib().orc_amax(_p(x, ctypes.c_float), x.size))


def global_scale(a) -> np.float32:
    """g = amax / (6 * 448)."""
    return np.float32(_lib().orc_global_scale(float(np.float32(a))))


def quantize(x, g=None) -> Q:
    """Activation quantisation (1x16 blocks along each row).  x: [R, C] FP32 values
    (BF16 inputs widened exactly).  g defaults to global_scale(amax(x))."""
    x = _f32(x)
    R, C = x.shape
    assert C % 16 == 0
    if g is None:
        g = global_scale(amax(x))
    codes = np.zeros((R, C // 2), np.uint8)
    scales = np.zeros((R, C // 16), np.uint8)
    _lib().orc_quant_rows(_p(x, ctypes.c_float), R, C, C, float(g),
                          _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8))
    return Q(codes, scales, np.float32(g), R, C)


def pack_weight(W):
    """Frozen weight W [N, K] -> (forward layout [N, K], backward layout [K, N]) with
    one E4M3 scale per 16x16 tile and one per-tensor g."""
    W = _f32(W)
    N, K = W.shape
    assert N % 16 == 0 and K % 16 == 0
    g = global_scale(amax(W))
    cf = np.zeros((N, K // 2), np.uint8)
    sf = np.zeros((N, K // 16), np.uint8)
    cb = np.zeros((K, N // 2), np.uint8)
    sb = np.zeros((K, N // 16), np.uint8)
    _lib().orc_pack_weight(_p(W, ctypes.c_float), N, K, float(g),
                           _p(cf, ctypes.c_uint8), _p(sf, ctypes.c_uint8),
                           _p(cb, ctypes.c_uint8), _p(sb, ctypes.c_uint8))
    return Q(cf, sf, g, N, K), Q(cb, sb, g, K, N)


def dequant(q: Q) -> np.ndarray:
    """Exact FP64 values e2m1(code) * e4m3(scale) * g."""
    out = np.empty((q.rows, q.cols), np.float64)
    codes = np.ascontiguousarray(q.codes)
    scales = np.ascontiguousarray(q.scales)
    _lib().orc_dequant_rows(_p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8),
                            float(q.g), q.rows, q.cols, _p(out, ctypes.c_double))
    return out


def dequant_rows(q: Q, rows) -> np.ndarray:
    """Exact FP64 dequantisation of a subset of rows (for sampled parity checks)."""
    rows = np.asarray(rows)
    sub = Q(np.ascontiguousarray(q.codes[rows]), np.ascontiguousarray(q.scales[rows]),
            q.g, len(rows), q.cols)
    return dequant(sub)


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """[R, C/2] bytes -> [R, C] 4-bit codes (even column from the low nibble)."""
    lo = codes & 0xF
    hi = codes >> 4
    out = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


# -------------------------------------------------- block-scaled MMA SF layout
def pad_to(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def sf_offset(r, c, c16p):
    """Byte offset of the scale of row r, block c in the 128x4-atom layout used by
    block-scaled tensor-core MMA: atoms of 128 rows x 4 blocks (512 bytes), ordered
    row-block major; inside an atom, byte (r%32)*16 + ((r%128)/32)*4 + c%4."""
    return (((r // 128) * (c16p // 4) + c // 4) * 512
            + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4))


def swizzle_scales(scales: np.ndarray) -> np.ndarray:
    """Logical [R, C16] scales -> flat [pad128(R) * pad4(C16)] bytes; pad bytes 0."""
    R, C16 = scales.shape
    Rp, C16p = pad_to(R, 128), pad_to(C16, 4)
    out = np.zeros(Rp * C16p, np.uint8)
    r = np.arange(R)[:, None]
    c = np.arange(C16)[None, :]
    out[sf_offset(r, c, C16p)] = scales
    return out


def unswizzle_scales(flat: np.ndarray, R: int, C16: int) -> np.ndarray:
    C16p = pad_to(C16, 4)
    r = np.arange(R)[:, None]
    c = np.arange(C16)[None, :]
    return np.asarray(flat).ravel()[sf_offset(r, c, C16p)]


# ----------------------------------------------------------------- LoRA linear
def lora_linear_fwd(xq: Q, wq_fwd: Q, A, B, alpha: float, residual=None, rows=None):
    """Y = Xhat Whatᵀ + (alpha/r) (Xhat A) B  [+ residual], FP64 (Table 7 rows
    "Frozen projections" and "LoRA branch"; Figure 3).  A [K, r], B [r, N] are the
    BF16 adapter values; Xhat, What are exactly dequantised.  rows: optional subset
    of output rows."""
    xh = dequant(xq) if rows is None else dequant_rows(xq, rows)
    wh = dequant(wq_fwd)
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    r = A.shape[1]
    y = xh @ wh.T + (alpha / r) * ((xh @ A) @ B)
    if residual is not None:
        res = np.asarray(residual, np.float64)
        y = y + (res if rows is None else res[rows])
    return y


def lora_linear_dgrad(dyq: Q, dy, wq_bwd: Q, A, B, alpha: float, dx_prev=None, rows=None):
    """dX = dYhat W + (alpha/r) (dY Bᵀ) Aᵀ  [+ dx_prev], FP64.  The frozen product
    uses the backward weight layout wq_bwd [K, N] (so dYhat @ wq_bwdᵀ); the LoRA
    input-gradient uses the BF16 dY (Table 7 "LoRA branch": BF16 input gradients)."""
    dyh = dequant(dyq) if rows is None else dequant_rows(dyq, rows)
    wb = dequant(wq_bwd)
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    dy64 = np.asarray(dy, np.float64)
    if rows is not None:
        dy64 = dy64[rows]
    r = A.shape[1]
    dx = dyh @ wb.T + (alpha / r) * ((dy64 @ B.T) @ A.T)
    if dx_prev is not None:
        p = np.asarray(dx_prev, np.float64)
        dx = dx + (p if rows is None else p[rows])
    return dx


def lora_adapter_grad(xq: Q, dy, A, B, alpha: float):
    """Gradients of the LoRA adapters of one LoRA linear, FP64 ("PACT: NVFP4
    Data-Flow LoRA Fine-Tuning on Consumer GPUs", Table 7 "LoRA branch": BF16 GEMMs
    on the reconstructed shared input; BF16 gradients).  With s = alpha / r,
    T = Xhat A and U = dY B^T:
        dA = s Xhat^T U   [K, r]      dB = s T^T dY   [r, N]
    Xhat is the exactly dequantised NVFP4 input the forward used; dY is the BF16
    gradient of the layer output (the values the dgrad's LoRA term also uses)."""
    xh = dequant(xq)
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    dy64 = np.asarray(dy, np.float64)
    s = alpha / A.shape[1]
    dA = s * (xh.T @ (dy64 @ B.T))
    dB = s * ((xh @ A).T @ dy64)
    return dA, dB


# ---------------------------------------------------------------- RMSNorm
EPS_DEFAULT = np.float32(1e-5)


def rmsnorm_fp32(x, gamma, eps=EPS_DEFAULT):
    """FP32 RMSNorm forward with the fixed reduction order; returns (rstd, y)."""
    x = _f32(x)
    gamma = _f32(gamma)
    R, H = x.shape
    assert H % 16 == 0
    rstd = np.empty(R, np.float32)
    y = np.empty((R, H), np.float32)
    _lib().orc_rmsnorm_rows(_p(x, ctypes.c_float), _p(gamma, ctypes.c_float), R, H,
                            float(np.float32(eps)), _p(rstd, ctypes.c_float),
                            _p(y, ctypes.c_float))
    return rstd, y


def rmsnorm_quant(x, gamma, eps=EPS_DEFAULT):
    """Fused RMSNorm -> NVFP4 (Table 7 "RMSNorm"): the FP32 output y is quantised
    directly (no BF16 rounding) with its own per-tensor scale.  Returns (yq, rstd)."""
    rstd, y = rmsnorm_fp32(x, gamma, eps)
    return quantize(y), rstd


def rmsnorm_bwd(yq: Q, gamma, rstd, dy, dres=None):
    """RMSNorm backward from the retained state (Table 7: FP32 reconstruction and
    reduction, BF16 gradient).  n = yhat / gamma, dn = dy * gamma,
    c = sum(dn * n) / H, dx = rstd * (dn - n * c)  [+ dres].  FP64."""
    dx = rmsnorm_bwd_from_y(dequant(yq), gamma, rstd, dy)
    if dres is not None:
        dx = dx + np.asarray(dres, np.float64)
    return dx


def rmsnorm_bwd_from_y(y, gamma, rstd, dy):
    """The RMSNorm input gradient given the (reconstructed) output y, FP64."""
    y = np.asarray(y, np.float64)
    g = np.asarray(gamma, np.float64)[None, :]
    n = y / g
    dn = np.asarray(dy, np.float64) * g
    H = y.shape[1]
    c = (dn * n).sum(axis=1, keepdims=True) / H
    return np.asarray(rstd, np.float64)[:, None] * (dn - n * c)


# ------------------------------------------------------------- exp and SiLU
def pexp(x) -> np.ndarray:
    x = _f32(x)
    flat = x.ravel()
    out = np.empty_like(flat)
    _lib().orc_pexp_array(_p(flat, ctypes.c_float), flat.size, _p(out, ctypes.c_float))
    return out.reshape(x.shape)


def silu_mul_fp32(gateup) -> np.ndarray:
    """h = (g / (1 + exp(-g))) * u in FP32 for gateup [M, 2I] (gate = columns [0, I),
    up = [I, 2I))."""
    gu = _f32(gateup)
    M, I2 = gu.shape
    I = I2 // 2
    h = np.empty((M, I), np.float32)
    _lib().orc_silu_mul_rows(_p(gu, ctypes.c_float), M, I, _p(h, ctypes.c_float))
    return h


def silu_mul_quant(gateup):
    """Fused SiLU-multiply -> NVFP4 (Table 7 "SiLU-multiply"): quantise h, and keep
    separate NVFP4 copies of gate and up, each with its own per-tensor scale.
    Returns (hq, gate_q, up_q)."""
    gu = _f32(gateup)
    I = gu.shape[1] // 2
    h = silu_mul_fp32(gu)
    return quantize(h), quantize(gu[:, :I]), quantize(gu[:, I:])


def silu_mul_bwd(gate_q: Q, up_q: Q, dh):
    """SiLU-multiply backward from the NVFP4 copies (Table 7: FP32 reconstruction and
    derivatives, BF16 gradients).  s = sigmoid(g):
      dgate = dh * u * s * (1 + g (1 - s)),  dup = dh * g * s.   FP64; [M, 2I]."""
    return silu_mul_bwd_from(dequant(gate_q), dequant(up_q), dh)


def silu_mul_bwd_from(g, u, dh):
    """SiLU-multiply gradients given (reconstructed) gate g and up u, FP64."""
    g = np.asarray(g, np.float64)
    u = np.asarray(u, np.float64)
    dh = np.asarray(dh, np.float64)
    s = 1.0 / (1.0 + np.exp(-g))
    dgate = dh * u * s * (1.0 + g * (1.0 - s))
    dup = dh * g * s
    return np.concatenate([dgate, dup], axis=1)


# ---------------------------------------------------------------- tolerance
def tol_bound(ref) -> np.ndarray:
    """Per-element acceptance bound for floating-point outputs:
    |gpu - ref| <= 8e-3 |ref| + 2e-3 rms(ref), rms over the whole reference tensor."""
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    return 8e-3 * np.abs(ref) + 2e-3 * rms


def check_close(gpu, ref, rms_ref=None):
    """Return (ok, worst_ratio, index); worst_ratio = max |gpu-ref| / bound."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    if rms_ref is None:
        bound = tol_bound(ref)
    else:
        bound = 8e-3 * np.abs(ref) + 2e-3 * rms_ref
    err = np.abs(gpu - ref)
    if err.size == 0:
        return True, 0.0, None
    ratio = err / np.maximum(bound, 1e-300)
    i = int(np.argmax(ratio))
    return bool(np.all(err <= bound)), float(ratio.ravel()[i]), np.unravel_index(i, err.shape)
