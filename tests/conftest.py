"""Shared pytest configuration.

Markers:
  gpu  -- needs a CUDA device and the compiled library; the CPU suite runs
          with ``-m "not gpu"``.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: test needs a CUDA device (B300) and the built library")
    config.addinivalue_line("markers", "slow: long-running test (full-size workloads)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.lib()
    return oracle
