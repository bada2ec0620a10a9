"""The debug build (libpact_debug.so: -DPACT_DEBUG, every kernel's hand-computed
store index checked against its buffer): a failing check is recorded in the device
status word and reported by pact_check_status instead of trapping, and the whole
guard-byte suite (one test per entry point) passes with that library loaded, with
no check failing."""
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


def test_guard_suite_under_the_debug_build(debug_env):
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu",
                        os.path.join(HERE, "test_gpu_canaries.py")],
                       env=debug_env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
