import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _no_wait_gave_up(request):
    """After every GPU test: no bounded wait of the library's kernels gave up during it (the
    poll synchronises the device and clears the count), so a pipeline stall is pinned to the
    test that caused it."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    import depth_wise_softmax_block_b300 as ar
    if ar._lib is None:
        return
    ar.attnres_poll_device_errors()
