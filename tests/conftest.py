import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (seconds to minutes)")


import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _ship_waits_never_gave_up(request):
    """After every GPU test: no bounded inbox wait of the ship kernel gave up."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    import cluster_distributed_shared_gb300 as pkg
    torch.cuda.synchronize()
    assert pkg.dsmem_hist_device_status() == 0, "a ship-kernel inbox wait timed out"
