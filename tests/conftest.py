"""Shared pytest configuration: the ``gpu`` marker and import paths."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled CUDA library")


def has_cuda() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def cuda_lib():
    """The compiled CUDA library binding; GPU tests fail loudly if it is missing."""
    if not has_cuda():
        pytest.fail("gpu test selected but no CUDA device is visible")
    import log_domain_sinkhorn_gb300 as lds
    return lds
