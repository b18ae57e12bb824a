import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


# One-line measured figures that GPU tests report (e.g. the free-running
# bf16 drift); printed in the terminal summary so they appear at the end of a
# quiet run.
_SUMMARY = []


@pytest.fixture
def summary_line():
    return _SUMMARY.append


def pytest_terminal_summary(terminalreporter):
    for line in _SUMMARY:
        terminalreporter.write_line(line)
