import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")


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


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


@pytest.fixture(autouse=True)
def _bounds_checks_held(request):
    """Under QSA_BOUNDS_CHECKED=1 (the bounds-checked library), every GPU test
    also asserts that no in-kernel bounds check failed while it ran."""
    yield
    if os.environ.get("QSA_BOUNDS_CHECKED", "") != "1" or "gpu" not in request.keywords:
        return
    import nvfp4_block_sparse_gb300 as qsa
    assert qsa.library_path().endswith("libqsa_bounds.so")
    code = qsa.qsa_debug_bounds_status()
    assert code == 0, "in-kernel bounds check failed: code 0x%x" % code
