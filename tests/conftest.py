import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a); runs the CUDA path through the C-ABI")
    config.addinivalue_line("markers", "slow: long-running (full-size workload)")


def pytest_collection_modifyitems(config, items):
    # keep the no-allocation entry point test last: pytest orders by file name
    # already; this only guards against plugins reordering
    items.sort(key=lambda it: 1 if "test_zz_" in it.nodeid else 0)
