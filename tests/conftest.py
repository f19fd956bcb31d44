import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


def pytest_collection_modifyitems(config, items):
    # GPU tests need CUDA; on a machine without a GPU they are skipped rather than failed
    # when selected explicitly with -m gpu.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def _cuda_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# Without a GPU the CUDA parity modules are not even imported (they load libfp8q.so and
# allocate device memory at import/fixture time); on a GPU machine a missing library fails loudly.
collect_ignore_glob = [] if _cuda_available() else ["test_gpu_*.py", "test_zz_*.py"]
