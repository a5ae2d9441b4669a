import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkvp.so")
    config.addinivalue_line("markers", "slow: long-running (large sizes)")


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


@pytest.fixture(autouse=True)
def _launch_options(request):
    """GPU tests run with programmatic dependent launch on, as the benchmark
    does (KVP_TEST_PDL=0 runs them with plain stream ordering)."""
    if "gpu" in request.keywords:
        import paged_prefix_reuse_gb300 as kvp

        if kvp._lib is not None:
            kvp.kvp_set_launch_options(kvp.LAUNCH_PDL if os.environ.get("KVP_TEST_PDL", "1") != "0" else 0)
    yield
