import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture(autouse=True)
def _guard_bands():
    """After each test, the guard bands around the device buffers it made are intact."""
    yield
    gpu_util = sys.modules.get("gpu_util")
    if gpu_util is not None and gpu_util._guarded:
        gpu_util.check_guards()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def read_golden(name):
    """Rows of a golden text fixture, '#' comment lines dropped."""
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]
