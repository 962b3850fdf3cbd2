import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library, on a GPU machine; builds it if needed."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from pmm_fc_layer_gb300 import build as _build
    _build.build()
    import pmm_fc_layer_gb300 as fc
    fc.load()
    return fc
