import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def read_golden(name):
    """Rows of a whitespace-separated fixture, comments and blank lines dropped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip() if line.lstrip().startswith("#") else line.strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def build_lib():
    """Build libfp8q.so if needed (loads the build script by path, since
    importing the package requires the built library)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("_fp8q_build", os.path.join(ROOT, "weight_transfer_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


@pytest.fixture(autouse=True)
def _no_device_errors(request):
    """After every GPU test: no kernel reported a copy that failed to land."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import weight_transfer_gb300 as w
    assert w.fp8q_device_errors(clear=True) == 0, "a kernel raised a device error flag"
