import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libcsa2.so")


def pytest_collection_modifyitems(config, items):
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


_check_handle = []


@pytest.fixture(autouse=True)
def _no_abandoned_wait(request):
    """After every GPU test: no bounded wait of the library's kernels gave up during it.  A wait
    that gives up records a code in a device error word and lets its kernel end, so the results
    after it mean nothing; csa2_check reads and clears the words (the failure-detection test
    provokes one on purpose and clears it itself)."""
    yield
    if "gpu" not in request.keywords:
        return
    import compressed_sparse_attention_03_gb300 as csa2

    if not _check_handle:
        _check_handle.append(csa2.csa2_create())
    assert csa2.csa2_check(_check_handle[0]) == 0, "a kernel's bounded wait gave up during this test"
