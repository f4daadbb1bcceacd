import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly when the device is missing; they are only skipped when the
    # caller explicitly deselects them with -m "not gpu".
    pass


@pytest.fixture(scope="session")
def golden():
    from tests.golden_io import load_golden
    return load_golden
