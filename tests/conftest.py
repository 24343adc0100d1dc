import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


@pytest.fixture(scope="session")
def rz():
    """The CUDA library binding; GPU tests only."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import invariant_logprobs_gb300 as rzmod
    rzmod.load()  # raises if the library is missing: no silent fallback
    return rzmod


@pytest.fixture(autouse=True)
def _device_bounds_checks(request):
    """With the debug build loaded (RZ_LIB_VARIANT=checks), every GPU test
    must leave no failed device bounds check behind."""
    yield
    if os.environ.get("RZ_LIB_VARIANT") != "checks" or "rz" not in request.fixturenames:
        return
    import invariant_logprobs_gb300 as rzmod
    res = rzmod.rz_debug_check_failures()
    assert res is not None, "RZ_LIB_VARIANT=checks but the loaded library has no checks"
    assert res[0] == 0, "failed device bounds checks: %d (first at site %d)" % res
