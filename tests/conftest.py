import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree; a GPU test fails (never skips) without it."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected but CUDA is not available")
    from paged_kv_cache_continuous_gb300 import binding
    return binding.load()
