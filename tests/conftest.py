"""Shared test set-up: repository root on sys.path, the ``gpu`` marker, and the oracle build."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on a GB300)")


@pytest.fixture(scope="session", autouse=True)
def _oracle_built():
    from oracle.build import build_oracle
    build_oracle()
