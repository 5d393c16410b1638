"""The C ABI from a plain C99 program (tests/cuda/abi_from_c.c): no Python,
torch or C++ between the caller and the library.

Without a GPU: both headers compile as strict C99 (gcc -std=c99 -pedantic
-Werror; the CUDA headers are system headers, exempt from -pedantic), the
program links against libnormfuse.so, and its host-side checks pass (bad
arguments rejected with the documented status, before any CUDA call).

With a GPU: the program allocates device memory itself, runs ln_fwd then
ln_bwd on inputs drawn by the seeded generators, and writes every output to
disk; the outputs are compared with the oracle under the tolerances of the
other parity tests.
"""

import glob
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import normalization_fwd_gb300 as nf
import workloads as W
from _parity import (amax_bits_of, check_elementwise, check_mean, check_rel, check_rel_l2,
                     dx_row_scale, oracle_bwd_rows, oracle_fwd)
from normalization_fwd_gb300 import build as nfbuild
from workloads import TORCH_DTYPES, as_f64, make_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "cuda", "abi_from_c.c")
DTYPE_CODE = {"f32": 0, "bf16": 1, "f16": 2}
MODE_CODE = {W.LAYERNORM: 0, W.RMSNORM: 1}


def _cuda_dirs():
    home = os.path.dirname(os.path.dirname(nfbuild.find_nvcc()))
    inc = os.path.join(home, "include")
    libs = [os.path.join(home, "lib64"), os.path.join(home, "lib")]
    libs += sorted(glob.glob(os.path.join(home, "targets", "*", "lib")))
    for d in libs:
        if glob.glob(os.path.join(d, "libcudart.so*")):
            return inc, d
    raise RuntimeError(f"libcudart.so not found under {home}")


@pytest.fixture(scope="module")
def c_program(tmp_path_factory):
    lib_path = nf.build_library()
    gcc = shutil.which("gcc") or shutil.which("cc")
    assert gcc, "no C compiler on PATH"
    inc, cudalib = _cuda_dirs()
    pkg = os.path.dirname(lib_path)
    out = str(tmp_path_factory.mktemp("abic") / "abi_from_c")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), "-isystem", inc, "-o", out, SRC,
           "-L", pkg, "-lnormfuse", f"-Wl,-rpath,{pkg}",
           "-L", cudalib, "-lcudart", f"-Wl,-rpath,{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


def test_headers_are_c99_and_host_checks_pass(c_program):
    r = subprocess.run([c_program, "check"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "check ok" in r.stdout


# Every operand present (bias, residual, beta), so the one C call path covers
# the whole block: aligned vectorised rows, an unaligned width that takes the
# scalar kernel, RMSNorm, and a ragged row count.
C_CASES = [
    W.LN_F32_4096x384.with_(name="c_ln_f32_300x384", rows=300),
    W.LN_F32_4096x384.with_(name="c_ln_bf16_129x1003", dtype="bf16", rows=129, hidden=1003),
    W.LN_F32_4096x384.with_(name="c_rms_bf16_200x2048", dtype="bf16", rows=200, hidden=2048,
                            mode=W.RMSNORM, beta_std=None),
    W.LN_F32_4096x384.with_(name="c_ln_f16_1000x4096", dtype="f16", rows=1000, hidden=4096,
                            x_std=3.0),
]


def _write(path, t):
    t.contiguous().view(torch.uint8).numpy().tofile(path)


def _read(path, dtype, shape):
    raw = np.fromfile(path, dtype=np.uint8)
    return torch.from_numpy(raw).view(dtype).reshape(shape)


@pytest.mark.gpu
@pytest.mark.parametrize("w", C_CASES, ids=lambda w: w.name)
def test_fwd_bwd_from_c_match_the_oracle(c_program, cuda_lib, w, tmp_path):
    inp = make_inputs(w, seed=5)
    dt = TORCH_DTYPES[w.dtype]
    R, H = w.rows, w.hidden
    beta = inp["beta"] if inp["beta"] is not None else torch.zeros(H, dtype=dt)
    for name, t in (("x", inp["x"]), ("bias", inp["bias"]), ("residual", inp["residual"]),
                    ("gamma", inp["gamma"]), ("beta", beta), ("dy", inp["dy"])):
        _write(tmp_path / f"{name}.bin", t)
    r = subprocess.run([c_program, "run", str(tmp_path), str(DTYPE_CODE[w.dtype]),
                        str(MODE_CODE[w.mode]), str(R), str(H), repr(w.eps)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr

    y = _read(tmp_path / "y.bin", dt, (R, H))
    s = _read(tmp_path / "sum.bin", dt, (R, H))
    dx = _read(tmp_path / "dx.bin", dt, (R, H))
    mean = _read(tmp_path / "mean.bin", torch.float32, (R,))
    rstd = _read(tmp_path / "rstd.bin", torch.float32, (R,))
    dgamma = _read(tmp_path / "dgamma.bin", torch.float32, (H,))
    dbeta = _read(tmp_path / "dbeta.bin", torch.float32, (H,))
    amax = _read(tmp_path / "amax.bin", torch.float32, (1,))

    ref = oracle_fwd(w, inp)
    check_elementwise(as_f64(s), ref["sum"], w.dtype, "sum", row_scale=False)
    check_elementwise(as_f64(y), ref["y_exact"], w.dtype, "y", row_scale=w.mode == W.LAYERNORM,
                      max_floored=1e-3)
    check_rel(as_f64(rstd), ref["rstd_exact"], 1e-5, "rstd")
    if w.mode == W.LAYERNORM:
        check_mean(as_f64(mean), ref["mean_exact"], ref["sum"])
    assert int(amax.numpy().view(np.uint32)[0]) == amax_bits_of(y)

    # The backward consumed the program's own forward outputs (sum, mean, rstd).
    m = mean if w.mode == W.LAYERNORM else None
    bref = oracle_bwd_rows(w, inp["dy"], s, inp["gamma"], m, rstd, slice(None))
    scale = dx_row_scale(as_f64(inp["dy"]), as_f64(inp["gamma"]), as_f64(rstd),
                         w.zero_centered_gamma)
    check_elementwise(as_f64(dx), bref["dx_exact"], w.dtype, "dx", scale_rows=scale,
                      max_floored=1e-3)
    check_rel_l2(as_f64(dgamma), bref["dgamma"], 1e-4, "dgamma")
    if w.mode == W.LAYERNORM:
        check_rel_l2(as_f64(dbeta), bref["dbeta"], 1e-4, "dbeta")
