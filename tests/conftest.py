import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def fgq():
    """The built library's Python binding (builds libfgq.so if needed)."""
    import fine_grained_fp8_gb300 as pkg
    from fine_grained_fp8_gb300 import build as fbuild
    fbuild.build()
    pkg.load()
    return pkg


@pytest.fixture(scope="session")
def cuda_dev(fgq):
    import torch
    assert torch.cuda.is_available(), "gpu tests need a CUDA device"
    return torch.device("cuda:0")
