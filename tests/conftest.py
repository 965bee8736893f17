import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # A gpu-marked test on a machine without a GPU fails loudly instead of
    # skipping: a skipped device test must not read as a pass.
    pass


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()
