import os
import sys

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU; runs the CUDA path")
    config.addinivalue_line("markers", "slow: full-size case")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle
