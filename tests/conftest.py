import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size case, minutes of CPU work for the oracle")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree. A GPU test without it fails loudly."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    from memory_bound_transformer_gb300 import capi
    return capi.load()
