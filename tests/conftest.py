import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Per-tensor worst errors of every value comparison against the FP64
    oracle in this run (max_abs with the scale its bar is taken relative
    to, and rel-L2), so the figures behind the tolerances are on record."""
    try:
        import _util
    except ImportError:  # pragma: no cover
        return
    if not _util.RECORDS:
        return
    terminalreporter.write_sep("-", "errors against the FP64 oracle (worst per tensor)")
    for line in _util.summary_lines():
        terminalreporter.write_line(line)
