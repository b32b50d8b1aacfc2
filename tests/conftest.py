"""Shared pytest set-up: the ``gpu`` marker and the repository on sys.path."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    """Skip GPU tests with a clear reason when no CUDA device is present."""
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """Write the per-call parity records (outputs beyond 1 ulp, exemptions) when LOWM_PARITY_LOG names a file."""
    try:
        import helpers
    except Exception:  # pragma: no cover
        return
    helpers.write_parity_log()
