"""Shared test set-up: the ``gpu`` marker, the repo root on sys.path, and
builders for the oracle (CPU, gcc) and the CUDA library (nvcc)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.build()
    return o
