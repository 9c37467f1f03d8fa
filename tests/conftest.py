import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libh3.so")
    config.addinivalue_line("markers", "slow: full-width shapes; minutes of CPU oracle time")


def pytest_collection_modifyitems(config, items):
    # GPU tests must fail loudly (not skip) when run on a box that has a GPU but
    # no library; on a CPU-only host they are deselected with -m "not gpu".
    pass


@pytest.fixture(scope="session")
def rng():
    import numpy as np
    return np.random.default_rng(1234)
