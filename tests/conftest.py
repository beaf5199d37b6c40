import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


def pytest_sessionstart(session):
    """Build libmoe.so when it is absent (a fresh checkout: the library is not versioned).
    An existing library is used as it is; `python -m quantized_moe_noaux_b300.build`
    rebuilds a stale one."""
    from quantized_moe_noaux_b300 import LIB_PATH
    if not os.path.exists(LIB_PATH):
        from quantized_moe_noaux_b300.build import build
        build()


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
