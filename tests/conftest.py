import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libk2")
    config.addinivalue_line("markers", "slow: full-size model parity (minutes of oracle time)")


def pytest_collection_modifyitems(config, items):
    # a gpu-marked test on a machine without a GPU is an error of the run, not a skip:
    # the driver runs `-m gpu` only where there is one.
    pass
