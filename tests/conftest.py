import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    # Keep the no-GPU suite honest: a gpu-marked test that somehow runs without
    # a GPU fails loudly instead of silently passing.
    pass


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    return oracle
