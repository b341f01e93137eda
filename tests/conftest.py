"""Shared pytest set-up: the ``gpu`` marker, the repo root on sys.path, and
session fixtures that build the oracle and the CUDA library on demand."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_built():
    from oracle import build
    return build.build()


@pytest.fixture(scope="session")
def lib_built():
    """The CUDA library, built in-tree if missing (nvcc cross-compiles without
    a GPU); CPU tests use only its host functions."""
    from sequence_head_relayout_gb300 import _build
    return _build.build()
