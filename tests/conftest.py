import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libpkv.so")
    config.addinivalue_line("markers", "slow: larger CPU cases")


def pytest_collection_modifyitems(config, items):
    # GPU tests are only meaningful with a device; without one they fail loudly
    # rather than silently skip, unless the run deselected them with -m "not gpu".
    pass


@pytest.fixture(scope="session")
def cuda_lib():
    """The product library with the CUDA path; fails loudly when absent."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    from paged_kv_cache_tables_gb300 import _binding
    return _binding.lib()
