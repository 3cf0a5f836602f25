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


def pytest_sessionfinish(session, exitstatus):
    """With KVQ_PARITY_REPORT=<path>, write every attention comparison's
    errors (plain max / mean against the stated bounds, the bf16 floor, the
    share of the allowance that is the binary32 bound) as JSON lines."""
    path = os.environ.get("KVQ_PARITY_REPORT")
    if not path:
        return
    mod = sys.modules.get("_harness")
    if mod is None:
        return
    import json
    REPORTS = mod.REPORTS
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "w") as f:
        for r in REPORTS:
            f.write(json.dumps(r) + "\n")
