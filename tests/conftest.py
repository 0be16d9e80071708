import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # a GPU-marked test on a machine without a GPU is skipped, never silently rerouted
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
def fa_lib():
    """The ctypes binding, building libfa_gb300.so first if it is missing."""
    lib_path = os.path.join(ROOT, "exact_tiled_attention_26_gb300", "libfa_gb300.so")
    if not os.path.exists(lib_path):
        import __graft_entry__
        __graft_entry__.build()
    import exact_tiled_attention_26_gb300 as fa
    return fa
