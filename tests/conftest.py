import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU work (full-size oracle runs)")


def pytest_collection_modifyitems(config, items):
    # Without a GPU every gpu-marked test is skipped rather than failed, so the
    # CPU suite stays green on build machines.
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


@pytest.fixture(autouse=True)
def _debug_build_bounds_clean(request):
    """With CONVFWD_DEBUG=1 (the debug build loaded), every GPU test must leave no
    out-of-range index in the device status word."""
    yield
    if "gpu" not in request.node.keywords or os.environ.get("CONVFWD_DEBUG", "") in ("", "0"):
        return
    import implicit_gemm_convolution_fwd_gb300 as cf
    if not cf.is_debug_build():
        return
    st = cf.device_status()
    assert not (st & cf.STATUS_BOUNDS_ANY), (
        f"debug build: an index fell outside its tensor (status {st:#x}, first index {cf.debug_first_bad_index()})")
