import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built library")
    config.addinivalue_line("markers", "slow: large CPU work")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (never skip into a fallback) when run without a GPU,
    # except when deselected with -m "not gpu".
    pass
