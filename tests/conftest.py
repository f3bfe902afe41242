import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda():
    """The CUDA device for GPU tests. Fails (never skips) when no GPU is visible, so that a box whose
    GPU is missing cannot report the CUDA path as tested."""
    import torch
    assert torch.cuda.is_available(), "GPU test run without a visible CUDA device"
    return torch.device("cuda:0")


def golden_path(name):
    return os.path.join(GOLDEN, name)


def read_golden(name):
    """Non-comment, non-empty lines of a golden fixture."""
    with open(golden_path(name)) as f:
        return [ln.rstrip("\n") for ln in f if ln.strip() and not ln.startswith("#")]
