import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU work (full-size oracle comparisons)")
    # enforced by the pytest-timeout plugin where it is installed; registered so that the mark
    # is known either way (tests that spawn processes also bound their own waits)
    config.addinivalue_line("markers", "timeout(seconds): upper bound on a test's run time")


def pytest_collection_modifyitems(config, items):
    have_gpu = False
    try:
        import torch

        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        pass
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
