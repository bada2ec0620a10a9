"""The C ABI library loads without a GPU and exports every function include/pact.h
declares; host-side argument checks reject bad calls before any launch."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pact.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pact_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from nvfp4_frozen_projection_gb300 import build
    path = build.build()
    return ctypes.CDLL(path), path


def test_header_declares_the_hot_path():
    names = set(_declared())
    for n in ("pact_quant_nvfp4", "pact_pack_weight_fwd", "pact_pack_weight_bwd",
              "pact_lora_linear_fwd", "pact_lora_linear_dgrad", "pact_lora_adapter_grad", "pact_rmsnorm_quant",
              "pact_silu_mul_quant", "pact_silu_mul_bwd", "pact_rmsnorm_bwd",
              "pact_check_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    so, path = lib
    for name in _declared():
        assert hasattr(so, name), f"{name} declared in pact.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(pact_[a-z0-9_]+)\b", out))
    assert set(_declared()) <= exported


def test_host_helpers_without_gpu(lib):
    so, _ = lib
    so.pact_nvfp4_sf_bytes.restype = ctypes.c_size_t
    so.pact_nvfp4_sf_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    so.pact_nvfp4_codes_bytes.restype = ctypes.c_size_t
    so.pact_nvfp4_codes_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    # Table 6: 4 bits per element + one byte per 16 elements (plus 128x4 padding)
    assert so.pact_nvfp4_codes_bytes(4096, 3072) == 4096 * 1536
    assert so.pact_nvfp4_sf_bytes(4096, 3072) == 4096 * 192
    assert so.pact_nvfp4_sf_bytes(1, 64) == 128 * 4
    so.pact_lora_linear_fwd_workspace_size.restype = ctypes.c_size_t
    so.pact_lora_linear_fwd_workspace_size.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_int]
    # LoRA left operand is a hi/lo BF16 pair (2 x 16 columns), right operand 16 columns,
    # and the transposed adapter A^T [16, K]
    assert so.pact_lora_linear_fwd_workspace_size(4096, 3072, 3072, 16) == 4096 * 64 + 3072 * 32 + 3072 * 32
    assert so.pact_lora_linear_fwd_workspace_size(4096, 3072, 3072, 65) == 0
    so.pact_version.restype = ctypes.c_char_p
    assert b"sm_103a" in so.pact_version()


def test_calls_fail_cleanly_without_device(lib):
    """With no usable CUDA device every entry point returns an error code (no crash)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    so, _ = lib
    so.pact_device_supported.restype = ctypes.c_int
    so.pact_last_error.restype = ctypes.c_char_p
    rc = so.pact_device_supported()
    assert rc != 0
    assert so.pact_last_error()
