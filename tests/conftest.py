import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300)")
    # compile the native parts if they are missing or stale (nvcc and gcc
    # work without a GPU); the package import fails loudly without them
    import __graft_entry__
    __graft_entry__.build()


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) on a machine without a GPU only when
    # the run did not ask for them explicitly with -m gpu.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
