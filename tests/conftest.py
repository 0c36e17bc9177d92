import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # A GPU test on a machine without a GPU is a hard failure when it is selected
    # explicitly with -m gpu; otherwise it is simply not selected.
    pass


@pytest.fixture(scope="session")
def root():
    return ROOT
