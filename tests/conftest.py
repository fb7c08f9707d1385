"""Shared pytest set-up: the ``gpu`` marker and access to the two libraries.

Tests marked ``gpu`` need a CUDA device and the sm_103a build of the CUDA
library; everything else runs on the CPU (the oracle, the host-side logic of
the library, the multi-process gloo paths).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the sm_103a CUDA library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def orc():
    """The CPU oracle (built on first use)."""
    import oracle
    oracle.lib()
    return oracle


def golden_path(name):
    return os.path.join(ROOT, "tests", "golden", name)
