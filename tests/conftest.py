"""Shared pytest setup: the `gpu` marker, import paths, and library builds.

Tests marked `gpu` need a CUDA device and call the CUDA library through its
C ABI; every other test runs on the CPU (the oracle's pins, the host-side
validation of the C ABI, the export table, the multi-process host logic).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (runs the CUDA library)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build.build()
    return oracle


@pytest.fixture(scope="session")
def rcc_lib():
    """The built C-ABI library (compiled here if it is missing or stale)."""
    from gradient_sync_rcc_gb300 import build as rbuild
    rbuild.build()
    from gradient_sync_rcc_gb300 import rcc
    return rcc


def cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False
