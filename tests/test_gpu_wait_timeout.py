"""Failure detection on the GPU without a fault: the bounded mbarrier wait
that every pipelined kernel uses gives up after its limit (about one second)
when the awaited copy never lands, reports it, and the context stays usable.

A small helper kernel (tests/cuda/wait_timeout.cu, compiled here with the
library's own bulk.cuh) waits on a barrier that nothing arrives at."""

import ctypes
import os
import shutil
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def helper(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = tmp_path_factory.mktemp("wt") / "libwait_timeout.so"
    src = os.path.join(ROOT, "tests", "cuda", "wait_timeout.cu")
    inc = os.path.join(ROOT, "normalization_fwd_gb300", "csrc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", "-I", inc, "-o", str(out), src], check=True)
    lib = ctypes.CDLL(str(out))
    lib.wait_timeout_launch.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.wait_timeout_launch.restype = ctypes.c_int
    return lib


def test_bounded_wait_gives_up_and_reports(helper, cuda_lib):
    torch.cuda.init()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    threads = 64
    assert helper.wait_timeout_launch(flag.data_ptr(), waited.data_ptr(), threads) == 0
    torch.cuda.synchronize()
    assert int(flag.item()) == threads            # every waiting thread gave up
    ns = int(waited.item())
    assert 0.9e9 <= ns <= 5e9, ns                  # after its ~1 s limit, not forever
    # the context is still usable: a normal call runs and is correct
    x = torch.randn(64, 384, device="cuda", dtype=torch.bfloat16)
    y = cuda_lib.softmax_fwd(x)
    torch.cuda.synchronize()
    assert torch.allclose(y.float().sum(dim=1), torch.ones(64, device="cuda"), atol=1e-2)
    assert cuda_lib.ln_device_error() == 0
