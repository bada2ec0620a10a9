"""The debug build (libpact_debug.so: -DPACT_DEBUG, every kernel's hand-computed
store index checked against its buffer, and the values that quantisations,
statistics and output amaxes read checked for NaN): a failing check is recorded in
the device status word and reported by pact_check_status instead of trapping, NaN
inputs are reported, and the whole guard-byte suite (one test per entry point)
passes with that library loaded, with no check failing."""
import os
import subprocess
import sys

import pytest

from nvfp4_frozen_projection_gb300 import build as pact_build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

PROBE = """
import nvfp4_frozen_projection_gb300 as pk
assert pk.library_path().endswith("libpact_debug.so"), pk.library_path()
assert "debug" in pk.pact_version(), pk.pact_version()
pk.pact_check_status()
pk.pact_test_bounds_check()
try:
    pk.pact_check_status()
except pk.PactError as e:
    assert e.code == 7 and "bounds" in str(e), (e.code, str(e))
else:
    raise SystemExit("the failing bounds check was not reported")
pk.pact_check_status()          # reading the word cleared it
print("debug status path ok")
"""

# One NaN in the values each kind of check covers: the per-block amax of every
# encoder, the weight amax, the RMSNorm statistic, the backward outputs and the GEMM
# epilogue (here through a NaN adapter value).  The debug library must report each
# as PACT_ERR_DEVICE_STATUS; finite inputs must leave the word clear.
NAN_CASES = """
import torch
import nvfp4_frozen_projection_gb300 as pk
dev = torch.device("cuda")
torch.manual_seed(0)
M, K, N, I, r = 200, 256, 192, 128, 12

def nan_at(t, idx):
    t = t.clone()
    t.view(-1)[idx] = float("nan")
    return t

def expect_nan(name, fn):
    pk.pact_check_status()
    fn()
    try:
        pk.pact_check_status()
    except pk.PactError as e:
        assert e.code == 7 and "NaN" in str(e), (name, e.code, str(e))
    else:
        raise SystemExit(name + ": a NaN input was not reported")

x = torch.randn(M, K, device=dev).bfloat16()
gamma = (1 + 0.1 * torch.randn(K, device=dev)).bfloat16()
gu = torch.randn(M, 2 * I, device=dev).bfloat16()
W = 0.05 * torch.randn(N, K, device=dev)
A = (torch.randn(K, r, device=dev) / K ** 0.5).bfloat16()
B = (0.1 * torch.randn(r, N, device=dev)).bfloat16()
dy = (0.1 * torch.randn(M, N, device=dev)).bfloat16()

# finite inputs: nothing recorded
xq = pk.pact_quant_nvfp4(x)
yq, rstd = pk.pact_rmsnorm_quant(x, gamma)
hq, gq, uq = pk.pact_silu_mul_quant(gu)
wf, wb = pk.pact_pack_weight_fwd(W), pk.pact_pack_weight_bwd(W)
pk.pact_lora_linear_fwd(xq, wf, A, B, 2.0)
pk.pact_lora_linear_dgrad_q(dy, wb, A, B, 2.0)
pk.pact_silu_mul_bwd(gq, uq, torch.randn(M, I, device=dev).bfloat16())
pk.pact_rmsnorm_bwd(yq, gamma, rstd, x)
pk.pact_check_status()

expect_nan("quant", lambda: pk.pact_quant_nvfp4(nan_at(x, 5 * K + 17)))
expect_nan("quant with a given amax",
           lambda: pk.pact_quant_nvfp4(nan_at(x, 77), amax=torch.ones(1, device=dev)))
expect_nan("rmsnorm_quant", lambda: pk.pact_rmsnorm_quant(nan_at(x, 3 * K + 1), gamma))
expect_nan("silu_mul_quant", lambda: pk.pact_silu_mul_quant(nan_at(gu, 2 * I + 3)))
expect_nan("pack_weight", lambda: pk.pact_pack_weight_fwd(nan_at(W, 40)))
expect_nan("fwd adapter", lambda: pk.pact_lora_linear_fwd(xq, wf, nan_at(A, 3), B, 2.0))
expect_nan("dgrad_q dY", lambda: pk.pact_lora_linear_dgrad_q(nan_at(dy, 9), wb, A, B, 2.0))
expect_nan("silu_mul_bwd", lambda: pk.pact_silu_mul_bwd(
    gq, uq, nan_at(torch.randn(M, I, device=dev).bfloat16(), 11)))
expect_nan("rmsnorm_bwd", lambda: pk.pact_rmsnorm_bwd(yq, gamma, rstd, nan_at(x, 13)))
print("NaN checks ok")
"""


@pytest.fixture(scope="module")
def debug_env():
    pact_build.build_debug()
    env = dict(os.environ, PACT_DEBUG="1")
    env["PYTHONPATH"] = os.pathsep.join(p for p in (ROOT, env.get("PYTHONPATH")) if p)
    return env


def test_release_build_compiles_the_checks_away():
    import nvfp4_frozen_projection_gb300 as pk
    if os.environ.get("PACT_DEBUG") == "1":
        pytest.skip("this process loaded the debug library")
    pk.pact_check_status()
    pk.pact_test_bounds_check()
    pk.pact_check_status()      # nothing recorded


def test_debug_build_reports_a_failed_check(debug_env):
    r = subprocess.run([sys.executable, "-c", PROBE], env=debug_env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]


def test_debug_build_reports_nan_inputs(debug_env):
    r = subprocess.run([sys.executable, "-c", NAN_CASES], env=debug_env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "NaN checks ok" in r.stdout


def test_release_build_does_not_look_for_nan():
    """The release library reads a NaN input without a status: its outputs are then
    unspecified, but the call ends and stays within its buffers."""
    import torch
    import nvfp4_frozen_projection_gb300 as pk
    if os.environ.get("PACT_DEBUG") == "1":
        pytest.skip("this process loaded the debug library")
    x = torch.randn(130, 256, device="cuda").bfloat16()
    x.view(-1)[7] = float("nan")
    pk.pact_check_status()
    pk.pact_quant_nvfp4(x)
    pk.pact_rmsnorm_quant(x, torch.ones(256, device="cuda").bfloat16())
    pk.pact_check_status()


def test_guard_suite_under_the_debug_build(debug_env):
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu",
                        os.path.join(HERE, "test_gpu_canaries.py")],
                       env=debug_env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
