import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the native library")


@pytest.fixture(scope="session")
def pages():
    with open(os.path.join(GOLDEN, "pages_figures.json")) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def native():
    """The native library (built in-tree on first use)."""
    from nvfp4_block_scaled_gather_gb300 import _native
    return _native.load()


@pytest.fixture(scope="session")
def cuda(native):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a visible CUDA device"
    return torch.device("cuda:0")
