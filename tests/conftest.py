"""Shared pytest configuration.

Tests marked ``gpu`` run the CUDA library on a GB300 and compare it with the
CPU oracle; everything else (oracle pins, host-side logic, the C-ABI symbol
table) runs on any machine.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built sm_103a library")


@pytest.fixture(scope="session")
def cuda_device():
    """The GPU the parity tests run on; fails (never skips) when there is none."""
    import torch

    assert torch.cuda.is_available(), "gpu-marked test run without a CUDA device"
    return torch.device("cuda:0")
