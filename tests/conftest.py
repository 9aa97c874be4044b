import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload cases")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def lib():
    """The CUDA library binding, built in-tree; the GPU tests call through its C-ABI."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_quantized_linear_gb300 import binding
    binding.load()
    return binding
