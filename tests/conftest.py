import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path)")


def pytest_sessionstart(session):
    # build (or bring up to date) libzp.so and the oracle before any import
    import __graft_entry__
    __graft_entry__._build_module().build()
    import oracle
    oracle.build()


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
