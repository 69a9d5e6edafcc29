"""Shared pytest configuration.

Tests marked ``gpu`` need a GB300 and the built CUDA library; everything else
runs on the CPU (the oracle against its pins, the library's host logic, the
exported C-ABI symbols, the multi-rank host paths over gloo).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")


def read_golden(name):
    """Rows of a golden fixture, comments and blank lines dropped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


@pytest.fixture
def golden():
    return read_golden


@pytest.fixture(params=["cxx", "numpy"])
def sim(request):
    """The oracle a pin runs against: the C++ simulation or the numpy one."""
    if request.param == "cxx":
        from oracle import cxx

        return cxx
    from oracle import schedules

    return schedules
