import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU test")


def pytest_collection_modifyitems(config, items):
    # the no-allocation entry point's test file must run last (it is collected last by
    # name); keep collection order otherwise
    items.sort(key=lambda it: os.path.basename(str(it.fspath)).startswith("test_zz_"))
