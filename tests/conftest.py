"""Shared pytest setup: the ``gpu`` marker and the repository on sys.path."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA device (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_device():
    """The CUDA device for -m gpu tests; missing CUDA is an error, not a skip."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test collected but torch.cuda.is_available() is False")
    return torch.device("cuda:0")
