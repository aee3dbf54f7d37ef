"""Shared pytest configuration: the ``gpu`` marker and build-on-demand of the CPU libraries."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libdg")


@pytest.fixture(scope="session", autouse=True)
def _built_cpu_libs():
    import dg_inputs
    import oracle
    dg_inputs.build()
    oracle.build()
    yield
