import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs through the C-ABI library)")


def pytest_collection_modifyitems(config, items):
    # A GPU test on a machine without CUDA fails loudly instead of skipping, so a
    # `-m gpu` run can never pass without having run the kernels.
    pass
