"""The kernel families that are not the default for a shape stay correct:
the parity files run again in child processes with the path switches set
(read once per process): NORMFUSE_FWD_PATH=ring (the pipelined forward
kernels), NORMFUSE_SMX_PATH=ring (the pipelined softmax kernels),
NORMFUSE_BWD_PATH=ring (the pipelined backward kernels also for the wide
rows that default to the register CTA-per-row backward) and
NORMFUSE_PATH=registers (the older register kernels, both directions)."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("env,files", [
    ({"NORMFUSE_FWD_PATH": "ring"}, ["tests/test_gpu_edges.py", "tests/test_gpu_fp8.py"]),
    ({"NORMFUSE_SMX_PATH": "ring"}, ["tests/test_gpu_softmax.py"]),
    ({"NORMFUSE_BWD_PATH": "ring"}, ["tests/test_gpu_edges.py", "tests/test_gpu_dbias.py"]),
    ({"NORMFUSE_PATH": "registers"}, ["tests/test_gpu_edges.py"]),
], ids=["fwd-ring", "softmax-ring", "bwd-ring", "registers"])
def test_parity_on_alternate_paths(cuda_lib, env, files):
    e = dict(os.environ)
    e.update(env)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
                        "-p", "no:cacheprovider", *files],
                       cwd=ROOT, env=e, capture_output=True, text=True, timeout=1200)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-15:])
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail
