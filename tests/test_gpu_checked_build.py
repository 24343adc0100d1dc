"""The debug build (-DRZ_CHECKS): every kernel checks its computed indices
against the call's sizes and records, instead of performing, any access that
would leave them.  This builds librz_checks.so and runs the odd-shape parity
suites against it in a child process (each test must pass and leave no
failed check); it also checks that the normal build reports having no
checks."""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu
SUITES = ["tests/test_gpu_parity.py", "tests/test_gpu_random_shapes.py",
          "tests/test_gpu_sampler.py", "tests/test_gpu_decode.py", "tests/test_gpu_profile.py"]


def test_normal_build_has_no_checks(rz):
    assert rz.rz_debug_check_failures() is None or \
        os.environ.get("RZ_LIB_VARIANT") == "checks"


@pytest.mark.skipif(os.environ.get("RZ_LIB_VARIANT") == "checks",
                    reason="already running under the debug build")
def test_odd_shapes_under_the_checked_build(rz):
    sys.path.insert(0, ROOT)
    from invariant_logprobs_gb300 import build
    build.build(checks=True)
    env = dict(os.environ, RZ_LIB_VARIANT="checks")
    p = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p",
                        "no:cacheprovider"] + SUITES, cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=1800)
    tail = (p.stdout + p.stderr)[-3000:]
    assert p.returncode == 0, tail
    assert " passed" in tail and "failed" not in tail, tail
