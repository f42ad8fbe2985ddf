"""Pytest configuration: the `gpu` marker and shared helpers.

Tests marked `gpu` need a CUDA device and the built CUDA library; everything
else runs on the CPU (the oracle pins, the host-side argument checks of the
C ABI, the multi-process host logic).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA device (B300) and the built libdsc.so")


@pytest.fixture(scope="session")
def oracle():
    import oracle as orc
    return orc
