import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_LIB = os.path.join(ROOT, "fsdp_sharded_optimizer_flatparameter_gb300", "libzs.so")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    # a fresh checkout has no libzs.so yet: build it once (nvcc, sm_103a) before the tests that load it;
    # a failed build raises here, so no test runs against a missing library
    if not os.path.exists(_LIB):
        path = os.path.join(ROOT, "fsdp_sharded_optimizer_flatparameter_gb300", "_build.py")
        spec = importlib.util.spec_from_file_location("_zs_build", path)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
