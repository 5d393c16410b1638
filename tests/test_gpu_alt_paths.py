"""The kernel families that are not the default for a shape stay correct:
the parity files run again in child processes whose calls the library plans
with the bulk-copy ring kernels, through its testing hook
ln_testing_select_kernels (the ``--ring-kernels`` option of the test suite):
the pipelined forward kernels, the pipelined softmax kernels, and the
pipelined backward kernels also for the wide rows that default to the
register CTA-per-row backward."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("ring,files", [
    ("forward", ["tests/test_gpu_edges.py", "tests/test_gpu_fp8.py"]),
    ("softmax", ["tests/test_gpu_softmax.py"]),
    ("backward", ["tests/test_gpu_edges.py", "tests/test_gpu_dbias.py"]),
], ids=["fwd-ring", "softmax-ring", "bwd-ring"])
def test_parity_on_alternate_paths(cuda_lib, ring, files):
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
                        "-p", "no:cacheprovider", f"--ring-kernels={ring}", *files],
                       cwd=ROOT, capture_output=True, text=True, timeout=1200)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-15:])
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail
