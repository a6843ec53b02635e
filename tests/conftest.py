import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (B300, sm_103a); parity tests through the C ABI")


def pytest_runtest_setup(item):
    # A GPU test must never pass silently on a machine without a GPU.
    if item.get_closest_marker("gpu") is not None:
        import torch
        if not torch.cuda.is_available():
            pytest.fail("gpu-marked test run without a CUDA device "
                        "(deselect with -m 'not gpu')", pytrace=False)
