import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads (several GB of inputs)")


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


@pytest.fixture(autouse=True)
def _device_error_word_is_clear_after_each_test(request):
    """With TREE_ATTN_CHECK_ERRORS set (the bounds-checking library's run, see
    test_debug_bounds_gpu.py), every GPU test must leave the device error word
    clear: a bounds error (or any device error a test did not expect and read
    back itself) fails the test that caused it."""
    yield
    if not os.environ.get("TREE_ATTN_CHECK_ERRORS") or "gpu" not in request.keywords:
        return
    import softmax_tree_reduction_gb300 as ta
    lib = ta.load()
    assert os.path.samefile(lib._name, os.environ["TREE_ATTN_LIBRARY"]), lib._name
    status = ta.tree_attn_get_device_error()
    assert status == 0, f"device error {status} ({ta.tree_attn_status_string(status)}) after {request.node.nodeid}"
