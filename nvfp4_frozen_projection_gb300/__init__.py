"""GB300-native NVFP4 LoRA linear (the hot path of PACT: "NVFP4 Data-Flow LoRA
Fine-Tuning on Consumer GPUs").

Thin Python binding over the C ABI of libpact (``include/pact.h``).  Every
function here has the same name as its C entry point and only marshals
arguments: torch provides device memory and the current stream, every step of
the computation runs in libpact's CUDA kernels.  There is no CPU fallback: if the
library is missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

__all__ = [
    "NVFP4", "PactError", "load_library", "library_path",
    "pact_quant_nvfp4", "pact_pack_weight_fwd", "pact_pack_weight_bwd",
    "pact_lora_linear_fwd", "pact_lora_linear_fwd_noalloc", "pact_lora_linear_dgrad",
    "pact_lora_linear_dgrad_q", "pact_lora_adapter_grad", "pact_rmsnorm_quant",
    "pact_silu_mul_quant", "pact_silu_mul_bwd", "pact_rmsnorm_bwd", "pact_test_pexp",
    "pact_pack_weight_fwd_gate_up", "pact_lora_linear_fwd_gate_up",
    "pact_test_wait_timeout", "pact_test_bounds_check", "pact_check_status",
    "pact_device_supported", "pact_launch_count", "pact_profile_next_gemm", "pact_version",
]

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    """libpact.so, or with PACT_DEBUG=1 in the environment the bounds-checked debug
    build libpact_debug.so (built by build.build_debug())."""
    if os.environ.get("PACT_DEBUG") == "1":
        return os.path.join(_HERE, "libpact_debug.so")
    return os.path.join(_HERE, "libpact.so")


class PactError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libpact error {code}: {msg}")
        self.code = code


class _NVFP4Struct(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("g", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


_LIB = None
_LIB_LOCK = threading.Lock()

_vp, _i64, _sz, _int, _f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
_SP = ctypes.POINTER(_NVFP4Struct)
_SIGNATURES = {
    "pact_nvfp4_codes_bytes": (_sz, [_i64, _i64]),
    "pact_nvfp4_sf_bytes": (_sz, [_i64, _i64]),
    "pact_quant_nvfp4_workspace_size": (_sz, [_i64, _i64]),
    "pact_quant_nvfp4": (_int, [_vp, _i64, _i64, _i64, _vp, _SP, _vp, _sz, _vp]),
    "pact_pack_weight_workspace_size": (_sz, [_i64, _i64]),
    "pact_pack_weight_fwd": (_int, [_vp, _i64, _i64, _SP, _vp, _sz, _vp]),
    "pact_pack_weight_bwd": (_int, [_vp, _i64, _i64, _SP, _vp, _sz, _vp]),
    "pact_pack_weight_fwd_gate_up": (_int, [_vp, _i64, _i64, _SP, _vp, _sz, _vp]),
    "pact_lora_linear_fwd_workspace_size": (_sz, [_i64, _i64, _i64, _int]),
    "pact_lora_linear_fwd": (_int, [_SP, _SP, _vp, _vp, _int, _f32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "pact_lora_linear_fwd_gate_up": (_int, [_SP, _SP, _vp, _vp, _int, _f32, _vp, _vp, _vp, _sz,
                                            _vp]),
    "pact_lora_linear_fwd_noalloc_max_scratch": (_sz, []),
    "pact_lora_linear_fwd_noalloc": (_int, [_SP, _SP, _vp, _vp, _int, _f32, _vp, _vp, _vp, _vp]),
    "pact_lora_linear_dgrad_workspace_size": (_sz, [_i64, _i64, _i64, _int]),
    "pact_lora_linear_dgrad": (_int, [_SP, _vp, _SP, _vp, _vp, _int, _f32, _int, _vp, _vp, _sz, _vp]),
    "pact_lora_linear_dgrad_q_workspace_size": (_sz, [_i64, _i64, _i64, _int]),
    "pact_lora_linear_dgrad_q": (_int, [_vp, _vp, _SP, _vp, _vp, _int, _f32, _int, _SP, _vp, _vp,
                                        _sz, _vp]),
    "pact_lora_adapter_grad_workspace_size": (_sz, [_i64, _i64, _i64, _int]),
    "pact_lora_adapter_grad": (_int, [_SP, _vp, _vp, _vp, _int, _f32, _i64, _vp, _vp, _vp, _sz, _vp]),
    "pact_rmsnorm_quant_workspace_size": (_sz, [_i64, _i64]),
    "pact_rmsnorm_quant": (_int, [_vp, _vp, _i64, _i64, _f32, _SP, _vp, _vp, _sz, _vp]),
    "pact_silu_mul_quant_workspace_size": (_sz, [_i64, _i64]),
    "pact_silu_mul_quant": (_int, [_vp, _i64, _i64, _vp, _SP, _SP, _SP, _vp, _sz, _vp]),
    "pact_silu_mul_bwd": (_int, [_SP, _SP, _vp, _vp, _vp, _vp]),
    "pact_rmsnorm_bwd": (_int, [_SP, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "pact_test_pexp": (_int, [_vp, _vp, _i64, _vp]),
    "pact_test_wait_timeout": (_int, [ctypes.c_uint32, _vp]),
    "pact_test_bounds_check": (_int, [_vp]),
    "pact_check_status": (_int, [_vp]),
    "pact_launch_count": (ctypes.c_uint64, []),
    "pact_profile_next_gemm": (_int, [_vp, _vp]),
    "pact_device_supported": (_int, []),
    "pact_last_error": (ctypes.c_char_p, []),
    "pact_version": (ctypes.c_char_p, []),
}


def load_library():
    """Load libpact.so (built in-tree by ``__graft_entry__.build()``)."""
    global _LIB
    with _LIB_LOCK:
        if _LIB is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"libpact.so is not built ({path}); run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _LIB = lib
    return _LIB


def _check(rc: int):
    if rc != 0:
        raise PactError(rc, load_library().pact_last_error().decode())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need_cuda(t: torch.Tensor, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------------ NVFP4 tensor
def _pad(x, m):
    return (x + m - 1) // m * m


@dataclass
class NVFP4:
    """Device NVFP4 tensor [rows, cols]: codes u8 [rows, cols/2], sf u8 (128x4-atom
    layout, pad128(rows) * pad4(cols/16) bytes), g f32 [1] (per-tensor scale)."""
    codes: torch.Tensor
    sf: torch.Tensor
    g: torch.Tensor
    rows: int
    cols: int

    @staticmethod
    def empty(rows: int, cols: int, device=None) -> "NVFP4":
        device = device or torch.device("cuda", torch.cuda.current_device())
        # 128-byte alignment of codes and sf comes from torch's caching allocator
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
        sf = torch.empty((_pad(rows, 128) * _pad(cols // 16, 4),), dtype=torch.uint8, device=device)
        g = torch.empty((1,), dtype=torch.float32, device=device)
        return NVFP4(codes, sf, g, rows, cols)

    def struct(self) -> _NVFP4Struct:
        return _NVFP4Struct(self.codes.data_ptr(), self.sf.data_ptr(), self.g.data_ptr(),
                            self.rows, self.cols)


# ------------------------------------------------------------------ workspace
_WS = {}


def _workspace(nbytes: int, device) -> torch.Tensor:
    """Per-(device, stream) scratch buffer, grown on demand.  Calls on one stream run
    in order, so they can share it."""
    key = (device.index if device.index is not None else torch.cuda.current_device(),
           torch.cuda.current_stream(device).cuda_stream)
    buf = _WS.get(key)
    need = max(256, int(nbytes))
    if buf is None or buf.numel() < need:
        buf = torch.empty((_pad(need, 1 << 20),), dtype=torch.uint8, device=device)
        _WS[key] = buf
    return buf


# ------------------------------------------------------------------ entry points
def pact_quant_nvfp4(x: torch.Tensor, amax: torch.Tensor | None = None,
                     out: NVFP4 | None = None) -> NVFP4:
    """Quantise BF16 x [M, K] (row stride may exceed K) to NVFP4."""
    lib = load_library()
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2):
        raise ValueError("x must be a 2-D CUDA bfloat16 tensor")
    if x.stride(1) != 1:
        raise ValueError("x must have unit column stride")
    M, K = x.shape
    out = out or NVFP4.empty(M, K, x.device)
    ws = _workspace(lib.pact_quant_nvfp4_workspace_size(M, K), x.device)
    s = out.struct()
    _check(lib.pact_quant_nvfp4(_ptr(x), M, K, x.stride(0), _ptr(amax), ctypes.byref(s),
                                _ptr(ws), ws.numel(), _stream()))
    return out


def _pack(W: torch.Tensor, backward: bool, out: NVFP4 | None, gate_up: bool = False) -> NVFP4:
    lib = load_library()
    _need_cuda(W, torch.float32, "W")
    N, K = W.shape
    out = out or (NVFP4.empty(K, N, W.device) if backward else NVFP4.empty(N, K, W.device))
    ws = _workspace(lib.pact_pack_weight_workspace_size(N, K), W.device)
    s = out.struct()
    fn = (lib.pact_pack_weight_bwd if backward else
          (lib.pact_pack_weight_fwd_gate_up if gate_up else lib.pact_pack_weight_fwd))
    _check(fn(_ptr(W), N, K, ctypes.byref(s), _ptr(ws), ws.numel(), _stream()))
    return out


def pact_pack_weight_fwd(W: torch.Tensor, out: NVFP4 | None = None) -> NVFP4:
    """Pack the frozen FP32 weight W [N, K] into the forward NVFP4 layout [N, K]."""
    return _pack(W, False, out)


def pact_pack_weight_bwd(W: torch.Tensor, out: NVFP4 | None = None) -> NVFP4:
    """Pack the frozen FP32 weight W [N, K] into the backward NVFP4 layout [K, N]."""
    return _pack(W, True, out)


def pact_pack_weight_fwd_gate_up(W: torch.Tensor, out: NVFP4 | None = None) -> NVFP4:
    """Forward pack of a fused gate|up weight [2I, K] in the interleaved row order that
    pact_lora_linear_fwd_gate_up reads."""
    return _pack(W, False, out, gate_up=True)


def pact_lora_linear_fwd_gate_up(xq: NVFP4, w_fwd_gu: NVFP4, A: torch.Tensor, B: torch.Tensor,
                                 scale: float, y: torch.Tensor | None = None,
                                 amax3: torch.Tensor | None = None):
    """The fused gate|up forward (y [M, 2I] as pact_lora_linear_fwd) and amax3 =
    (max |silu(gate) up|, max |gate|, max |up|) of it.  Returns (y, amax3)."""
    lib = load_library()
    _need_cuda(A, torch.bfloat16, "A")
    _need_cuda(B, torch.bfloat16, "B")
    M, K, N = xq.rows, xq.cols, w_fwd_gu.rows
    r = A.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if amax3 is None:
        amax3 = torch.empty(3, dtype=torch.float32, device=A.device)
    _need_cuda(y, torch.bfloat16, "y")
    _need_cuda(amax3, torch.float32, "amax3")
    ws = _workspace(lib.pact_lora_linear_fwd_workspace_size(M, N, K, r), A.device)
    sx, sw = xq.struct(), w_fwd_gu.struct()
    _check(lib.pact_lora_linear_fwd_gate_up(ctypes.byref(sx), ctypes.byref(sw), _ptr(A), _ptr(B), r,
                                            float(scale), _ptr(y), _ptr(amax3), _ptr(ws),
                                            ws.numel(), _stream()))
    return y, amax3


def pact_lora_linear_fwd(xq: NVFP4, w_fwd: NVFP4, A: torch.Tensor, B: torch.Tensor,
                         scale: float, residual: torch.Tensor | None = None,
                         y: torch.Tensor | None = None,
                         out_amax: torch.Tensor | None = None) -> torch.Tensor:
    """Y = Xhat What^T + scale (Xhat A) B [+ residual], BF16 [M, N]."""
    lib = load_library()
    _need_cuda(A, torch.bfloat16, "A")
    _need_cuda(B, torch.bfloat16, "B")
    M, K, N = xq.rows, xq.cols, w_fwd.rows
    r = A.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need_cuda(y, torch.bfloat16, "y")
    if residual is not None:
        _need_cuda(residual, torch.bfloat16, "residual")
    ws = _workspace(lib.pact_lora_linear_fwd_workspace_size(M, N, K, r), A.device)
    sx, sw = xq.struct(), w_fwd.struct()
    _check(lib.pact_lora_linear_fwd(ctypes.byref(sx), ctypes.byref(sw), _ptr(A), _ptr(B), r,
                                    float(scale), _ptr(residual), _ptr(y), _ptr(out_amax),
                                    _ptr(ws), ws.numel(), _stream()))
    return y


def pact_lora_linear_fwd_noalloc(xq: NVFP4, w_fwd: NVFP4, A: torch.Tensor, B: torch.Tensor,
                                 scale: float, y: torch.Tensor,
                                 residual: torch.Tensor | None = None,
                                 out_amax: torch.Tensor | None = None) -> torch.Tensor:
    """pact_lora_linear_fwd for callers that cannot allocate: the output y is
    preallocated by the caller and the library's fixed scratch array replaces the
    workspace (calls that overlap on the GPU race on it)."""
    lib = load_library()
    _need_cuda(A, torch.bfloat16, "A")
    _need_cuda(B, torch.bfloat16, "B")
    _need_cuda(y, torch.bfloat16, "y")
    sx, sw = xq.struct(), w_fwd.struct()
    _check(lib.pact_lora_linear_fwd_noalloc(ctypes.byref(sx), ctypes.byref(sw), _ptr(A), _ptr(B),
                                            A.shape[1], float(scale), _ptr(residual), _ptr(y),
                                            _ptr(out_amax), _stream()))
    return y


def pact_lora_linear_dgrad(dyq: NVFP4, dy: torch.Tensor, w_bwd: NVFP4, A: torch.Tensor,
                           B: torch.Tensor, scale: float, dx: torch.Tensor | None = None,
                           accumulate: bool = False) -> torch.Tensor:
    """dX = dYhat W + scale (dY B^T) A^T [+ dX if accumulate], BF16 [M, K]."""
    lib = load_library()
    _need_cuda(dy, torch.bfloat16, "dy")
    _need_cuda(A, torch.bfloat16, "A")
    _need_cuda(B, torch.bfloat16, "B")
    M, N, K = dyq.rows, dyq.cols, w_bwd.rows
    r = A.shape[1]
    if dx is None:
        if accumulate:
            raise ValueError("accumulate needs dx")
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device)
    _need_cuda(dx, torch.bfloat16, "dx")
    ws = _workspace(lib.pact_lora_linear_dgrad_workspace_size(M, N, K, r), dy.device)
    sd, sw = dyq.struct(), w_bwd.struct()
    _check(lib.pact_lora_linear_dgrad(ctypes.byref(sd), _ptr(dy), ctypes.byref(sw), _ptr(A),
                                      _ptr(B), r, float(scale), int(bool(accumulate)), _ptr(dx),
                                      _ptr(ws), ws.numel(), _stream()))
    return dx


def pact_lora_linear_dgrad_q(dy: torch.Tensor, w_bwd: NVFP4, A: torch.Tensor, B: torch.Tensor,
                             scale: float, amax: torch.Tensor | None = None,
                             dyq: NVFP4 | None = None, dx: torch.Tensor | None = None,
                             accumulate: bool = False):
    """Quantise dY into dyq and run the LoRA-linear input gradient in one call:
    the same results as pact_quant_nvfp4 + pact_lora_linear_dgrad.  Returns (dx, dyq)."""
    lib = load_library()
    _need_cuda(dy, torch.bfloat16, "dy")
    _need_cuda(A, torch.bfloat16, "A")
    _need_cuda(B, torch.bfloat16, "B")
    M, N = dy.shape
    K = w_bwd.rows
    r = A.shape[1]
    if amax is not None:
        _need_cuda(amax, torch.float32, "amax")
    if dyq is None:
        dyq = NVFP4.empty(M, N, dy.device)
    if dx is None:
        if accumulate:
            raise ValueError("accumulate needs dx")
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device)
    _need_cuda(dx, torch.bfloat16, "dx")
    ws = _workspace(lib.pact_lora_linear_dgrad_q_workspace_size(M, N, K, r), dy.device)
    sq, sw = dyq.struct(), w_bwd.struct()
    _check(lib.pact_lora_linear_dgrad_q(_ptr(dy), _ptr(amax), ctypes.byref(sw), _ptr(A), _ptr(B),
                                        r, float(scale), int(bool(accumulate)), ctypes.byref(sq),
                                        _ptr(dx), _ptr(ws), ws.numel(), _stream()))
    return dx, dyq


def pact_lora_adapter_grad(xq: NVFP4, dy: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                           scale: float, dA: torch.Tensor | None = None,
                           dB: torch.Tensor | None = None):
    """dA = scale Xhat^T (dY B^T) FP32 [K, r] and dB = scale (Xhat A)^T dY FP32 [r, N]."""
    lib = load_library()
    _need_cuda(dy, torch.bfloat16, "dy")
    _need_cuda(A, torch.bfloat16, "A")
    _need_cuda(B, torch.bfloat16, "B")
    M, K = xq.rows, xq.cols
    N = dy.shape[1]
    r = A.shape[1]
    if dA is None:
        dA = torch.empty((K, r), dtype=torch.float32, device=dy.device)
    if dB is None:
        dB = torch.empty((r, N), dtype=torch.float32, device=dy.device)
    _need_cuda(dA, torch.float32, "dA")
    _need_cuda(dB, torch.float32, "dB")
    ws = _workspace(lib.pact_lora_adapter_grad_workspace_size(M, N, K, r), dy.device)
    sx = xq.struct()
    _check(lib.pact_lora_adapter_grad(ctypes.byref(sx), _ptr(dy), _ptr(A), _ptr(B), r,
                                      float(scale), N, _ptr(dA), _ptr(dB), _ptr(ws), ws.numel(),
                                      _stream()))
    return dA, dB


def pact_rmsnorm_quant(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-5,
                       out: NVFP4 | None = None, rstd: torch.Tensor | None = None):
    """Fused RMSNorm -> NVFP4.  Returns (yq, rstd)."""
    lib = load_library()
    _need_cuda(x, torch.bfloat16, "x")
    _need_cuda(gamma, torch.bfloat16, "gamma")
    M, H = x.shape
    out = out or NVFP4.empty(M, H, x.device)
    if rstd is None:
        rstd = torch.empty((M,), dtype=torch.float32, device=x.device)
    ws = _workspace(lib.pact_rmsnorm_quant_workspace_size(M, H), x.device)
    s = out.struct()
    _check(lib.pact_rmsnorm_quant(_ptr(x), _ptr(gamma), M, H, float(eps), ctypes.byref(s),
                                  _ptr(rstd), _ptr(ws), ws.numel(), _stream()))
    return out, rstd


def pact_silu_mul_quant(gateup: torch.Tensor, amax3: torch.Tensor | None = None,
                        outs: tuple | None = None):
    """Fused SiLU-multiply -> NVFP4 on gateup [M, 2I].  Returns (hq, gate_q, up_q)."""
    lib = load_library()
    _need_cuda(gateup, torch.bfloat16, "gateup")
    M, I2 = gateup.shape
    I = I2 // 2
    hq, gq, uq = outs or tuple(NVFP4.empty(M, I, gateup.device) for _ in range(3))
    ws = _workspace(lib.pact_silu_mul_quant_workspace_size(M, I), gateup.device)
    sh, sg, su = hq.struct(), gq.struct(), uq.struct()
    _check(lib.pact_silu_mul_quant(_ptr(gateup), M, I, _ptr(amax3), ctypes.byref(sh),
                                   ctypes.byref(sg), ctypes.byref(su), _ptr(ws), ws.numel(),
                                   _stream()))
    return hq, gq, uq


def pact_silu_mul_bwd(gate_q: NVFP4, up_q: NVFP4, dh: torch.Tensor,
                      dgateup: torch.Tensor | None = None,
                      out_amax: torch.Tensor | None = None) -> torch.Tensor:
    """SiLU-multiply backward from the NVFP4 gate/up copies.  Returns dgateup [M, 2I]."""
    lib = load_library()
    _need_cuda(dh, torch.bfloat16, "dh")
    M, I = gate_q.rows, gate_q.cols
    if dgateup is None:
        dgateup = torch.empty((M, 2 * I), dtype=torch.bfloat16, device=dh.device)
    sg, su = gate_q.struct(), up_q.struct()
    _check(lib.pact_silu_mul_bwd(ctypes.byref(sg), ctypes.byref(su), _ptr(dh), _ptr(dgateup),
                                 _ptr(out_amax), _stream()))
    return dgateup


def pact_rmsnorm_bwd(yq: NVFP4, gamma: torch.Tensor, rstd: torch.Tensor, dy: torch.Tensor,
                     dres: torch.Tensor | None = None,
                     dx: torch.Tensor | None = None,
                     out_amax: torch.Tensor | None = None) -> torch.Tensor:
    """RMSNorm backward from the retained NVFP4 output and rstd [+ dres].  out_amax
    (FP32 [1], optional) receives max |dx| for a single-pass quantisation of dx."""
    lib = load_library()
    _need_cuda(dy, torch.bfloat16, "dy")
    if dx is None:
        dx = torch.empty_like(dy)
    if out_amax is not None:
        _need_cuda(out_amax, torch.float32, "out_amax")
    s = yq.struct()
    _check(lib.pact_rmsnorm_bwd(ctypes.byref(s), _ptr(gamma), _ptr(rstd), _ptr(dy), _ptr(dres),
                                _ptr(dx), _ptr(out_amax), _stream()))
    return dx


def pact_test_pexp(x: torch.Tensor) -> torch.Tensor:
    """The FP32 exp recipe used inside the SiLU kernels, element-wise on the GPU."""
    lib = load_library()
    _need_cuda(x, torch.float32, "x")
    y = torch.empty_like(x)
    _check(lib.pact_test_pexp(_ptr(x), _ptr(y), x.numel(), _stream()))
    return y


def pact_test_wait_timeout(limit_us: int = 1000) -> None:
    """Launch a kernel whose bounded wait runs out after limit_us microseconds; the
    next pact_check_status() raises PactError with code PACT_ERR_TIMEOUT (6)."""
    _check(load_library().pact_test_wait_timeout(int(limit_us), _stream()))


def pact_test_bounds_check() -> None:
    """Evaluate one failing bounds check on the GPU (no memory access): with the debug
    library the next pact_check_status() raises PactError (PACT_ERR_DEVICE_STATUS);
    with the release library it passes."""
    _check(load_library().pact_test_bounds_check(_stream()))


def pact_version() -> str:
    return load_library().pact_version().decode()


def pact_check_status() -> None:
    """Synchronise the current stream and raise if a kernel recorded an error."""
    _check(load_library().pact_check_status(_stream()))


def pact_device_supported() -> bool:
    return load_library().pact_device_supported() == 0


def pact_launch_count() -> int:
    """Number of libpact kernels launched by this process so far."""
    return int(load_library().pact_launch_count())


def pact_profile_next_gemm(begin: torch.cuda.Event, end: torch.cuda.Event) -> None:
    """Record begin/end on the launch stream around the next NVFP4 GEMM kernel."""
    _check(load_library().pact_profile_next_gemm(ctypes.c_void_p(begin.cuda_event),
                                                 ctypes.c_void_p(end.cuda_event)))
