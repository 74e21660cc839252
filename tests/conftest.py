import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libdd.so")
    config.addinivalue_line("markers", "slow: long-running (full-size parity)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session", autouse=True)
def _built_library():
    """Compile libdd.so (nvcc, sm_103a) if it is missing or stale."""
    from sparse_kv_prefetch_gb300 import build
    build.ensure_built()


@pytest.fixture(autouse=True)
def _release_memory(request):
    """After every GPU test: free cached device memory and the page-locked host
    blocks torch keeps for reuse, so the full-size cases (host stores of up to
    96 GiB) never add up on the host."""
    yield
    if "gpu" not in request.keywords:
        return
    import gc

    import torch
    gc.collect()
    if torch.cuda.is_available() and torch.cuda.is_initialized():
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        if hasattr(torch._C, "_host_emptyCache"):
            torch._C._host_emptyCache()
