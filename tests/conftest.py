"""Shared pytest configuration.

Tests marked ``gpu`` need an sm_103 GPU and the built CUDA library; every
other test runs on the CPU.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs an sm_103 GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity cases")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN
