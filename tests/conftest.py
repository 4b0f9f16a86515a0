import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built libmxq.so")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(autouse=True)
def _gpu_tests_need_a_device(request):
    """A GPU test on a host without a CUDA device fails instead of skipping,
    so a run of `-m gpu` that could not reach the kernels never passes."""
    if request.node.get_closest_marker("gpu") is not None:
        import torch

        if not torch.cuda.is_available():
            pytest.fail("GPU test without a CUDA device")
