"""GPU parity on seeded random shapes: dtype, rows, hidden (16-byte multiples
more often than not, so every vector layout is reached, and odd widths for
the scalar kernels), mode, zero-centered gamma, optional bias / residual /
beta and dbias, all drawn from one fixed seed. Each case runs the forward
and the backward against the oracle with the tolerances of the other
parity tests."""

import numpy as np
import pytest
import torch

import workloads as W
from _parity import (amax_bits_got, amax_bits_of, check_elementwise, check_mean, check_rel,
                     check_rel_l2, dx_row_scale, gpu_bwd, gpu_fwd, oracle_bwd_rows, oracle_fwd)
from workloads import Workload, as_f64, make_inputs

pytestmark = pytest.mark.gpu


def _cases(n=40, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = ["bf16", "f16", "f32"][rng.integers(3)]
        vec = 16 // (4 if dtype == "f32" else 2)
        top = 8192 if dtype == "f32" else 16384
        hidden = int(np.exp(rng.uniform(0.0, np.log(top))))
        if rng.random() < 0.7:
            hidden = max(vec, hidden // vec * vec)
        hidden = max(1, min(hidden, top))
        rows = int(rng.integers(1, 3000)) if hidden <= 4096 else int(rng.integers(1, 600))
        mode = W.RMSNORM if rng.random() < 0.5 else W.LAYERNORM
        w = Workload(name=f"rand{i}_{dtype}_{rows}x{hidden}_{mode}", dtype=dtype, rows=rows,
                     hidden=hidden, mode=mode, eps=float(10.0 ** rng.uniform(-6, -4)),
                     x_std=float(rng.uniform(0.5, 3.0)),
                     residual_std=1.0 if rng.random() < 0.7 else None,
                     bias_std=0.2 if rng.random() < 0.5 else None,
                     gamma_std=0.2,
                     beta_std=(0.2 if rng.random() < 0.8 else None) if mode == W.LAYERNORM else None,
                     zero_centered_gamma=bool(rng.random() < 0.3), amax=True)
        out.append((w, bool(rng.random() < 0.5)))
    return out


CASES = _cases()


@pytest.mark.parametrize("w,dbias", CASES, ids=[c[0].name for c in CASES])
def test_random_shape_matches_oracle(cuda_lib, w, dbias):
    inp = make_inputs(w, seed=w.rows * 7 + w.hidden)
    ref = oracle_fwd(w, inp)
    got = gpu_fwd(cuda_lib, w, inp)
    assert got["guards_ok"]
    if "sum" in got:
        check_elementwise(as_f64(got["sum"]), ref["sum"], w.dtype, "sum", row_scale=False)
    check_elementwise(as_f64(got["y"]), ref["y_exact"], w.dtype, "y",
                      row_scale=w.mode == W.LAYERNORM)
    check_rel(as_f64(got["rstd"]), ref["rstd_exact"], 1e-5, "rstd")
    if w.mode == W.LAYERNORM:
        check_mean(as_f64(got["mean"]), ref["mean_exact"], ref["sum"])
    assert amax_bits_got(got["amax"]) == amax_bits_of(got["y"])

    dt = W.TORCH_DTYPES[w.dtype]
    x_sum = torch.from_numpy(ref["sum"]).to(dt)
    mean = None if ref["mean"] is None else torch.from_numpy(ref["mean"]).float()
    rstd = torch.from_numpy(ref["rstd"]).float()
    bref = oracle_bwd_rows(w, inp["dy"], x_sum, inp["gamma"], mean, rstd, slice(None))
    bgot = gpu_bwd(cuda_lib, w, inp["dy"], x_sum, inp["gamma"], mean, rstd, need_dbias=dbias)
    assert bgot["guards_ok"]
    scale = dx_row_scale(as_f64(inp["dy"]), as_f64(inp["gamma"]), as_f64(rstd),
                         w.zero_centered_gamma)
    check_elementwise(as_f64(bgot["dx"]), bref["dx_exact"], w.dtype, "dx", scale_rows=scale)
    check_rel_l2(as_f64(bgot["dgamma"]), bref["dgamma"], 1e-4, "dgamma")
    if w.mode == W.LAYERNORM:
        check_rel_l2(as_f64(bgot["dbeta"]), bref["dbeta"], 1e-4, "dbeta")
    if dbias:
        check_rel_l2(as_f64(bgot["dbias"]), bref["dbias"], 1e-4, "dbias")
