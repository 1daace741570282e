"""pytest configuration: the `gpu` marker and shared helpers.

Tests marked `gpu` need a CUDA device and the compiled sm_103a library; all
other tests run on CPU only.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled sm_103a library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
