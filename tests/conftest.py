import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA library through its C ABI")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree; the GPU tests fail loudly without it."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    import normalization_fwd_gb300 as nf
    nf.load_library()
    return nf
