import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")


def pytest_collection_modifyitems(config, items):
    # Fail loudly instead of silently skipping: a gpu test run without a GPU is an error,
    # but plain CPU runs select them out with -m "not gpu".
    pass


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()
