import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption(
        "--ring-kernels", default="",
        help="comma-separated directions (forward, backward, softmax) whose calls the GPU "
             "tests plan with the bulk-copy ring kernels instead of the default ones "
             "(through the library's testing hook ln_testing_select_kernels)")


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA library through its C ABI")


@pytest.fixture(scope="session")
def cuda_lib(request):
    """The CUDA library, built in-tree; the GPU tests fail loudly without it."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    import normalization_fwd_gb300 as nf
    nf.load_library()
    ring = {d for d in request.config.getoption("--ring-kernels").split(",") if d}
    unknown = ring - {"forward", "backward", "softmax"}
    if unknown:
        pytest.fail(f"--ring-kernels: unknown direction(s) {sorted(unknown)}")
    fam = {d: ("ring" if d in ring else "default") for d in ("forward", "backward", "softmax")}
    nf.ln_testing_select_kernels(**fam)
    return nf
