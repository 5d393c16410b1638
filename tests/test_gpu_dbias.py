"""GPU parity of the bias gradient (ln_bwd_ex): dbias = sum over rows of dx,
the third column reduction fused into the backward's persistent kernel.

Checked against the oracle's dbias (fp32 rules: relative L2 <= 1e-4); dx,
dgamma and dbeta against the oracle with the usual tolerances. (With dbias a
shape can run on another kernel family than ln_bwd does, e.g. CTA-per-row
where ln_bwd uses lane groups, so dx need not be bitwise that of ln_bwd.)
"""

import numpy as np
import pytest
import torch

import workloads as W
from _parity import (check_elementwise, check_rel_l2, dx_row_scale, gpu_bwd, oracle_bwd_rows,
                     oracle_fwd)
from workloads import Workload, as_f64, make_inputs

pytestmark = pytest.mark.gpu


def wl(dtype, rows, hidden, mode):
    return Workload(name=f"dbias_{dtype}_{rows}x{hidden}_{mode}", dtype=dtype, rows=rows,
                    hidden=hidden, mode=mode, eps=1e-5, x_std=1.0, residual_std=1.0,
                    bias_std=0.1, gamma_std=0.1,
                    beta_std=0.1 if mode == W.LAYERNORM else None)


@pytest.mark.parametrize("mode", [W.LAYERNORM, W.RMSNORM])
@pytest.mark.parametrize("dtype,rows,hidden", [
    ("bf16", 20001, 384),      # lane-group pipelined kernel
    ("f16", 4099, 1280),
    ("f32", 3001, 768),
    ("bf16", 601, 8192),       # CTA-per-row pipelined kernel
    ("bf16", 777, 1001),       # scalar kernel
])
def test_dbias_matches_oracle(cuda_lib, dtype, rows, hidden, mode):
    w = wl(dtype, rows, hidden, mode)
    inp = make_inputs(w, seed=11)
    ref = oracle_fwd(w, inp)
    dt = W.TORCH_DTYPES[w.dtype]
    x_sum = torch.from_numpy(ref["sum"]).to(dt)
    mean = None if ref["mean"] is None else torch.from_numpy(ref["mean"]).float()
    rstd = torch.from_numpy(ref["rstd"]).float()
    bref = oracle_bwd_rows(w, inp["dy"], x_sum, inp["gamma"], mean, rstd, slice(None))
    ex = gpu_bwd(cuda_lib, w, inp["dy"], x_sum, inp["gamma"], mean, rstd, need_dbias=True)
    assert ex["guards_ok"]
    check_rel_l2(as_f64(ex["dbias"]), bref["dbias"], 1e-4, "dbias")
    check_elementwise(as_f64(ex["dx"]), bref["dx_exact"], dtype, "dx",
                      scale_rows=dx_row_scale(as_f64(inp["dy"]), as_f64(inp["gamma"]),
                                              as_f64(rstd), w.zero_centered_gamma))
    check_rel_l2(as_f64(ex["dgamma"]), bref["dgamma"], 1e-4, "dgamma")
    if mode == W.LAYERNORM:
        check_rel_l2(as_f64(ex["dbeta"]), bref["dbeta"], 1e-4, "dbeta")


@pytest.mark.parametrize("gdt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("mode", [W.LAYERNORM, W.RMSNORM])
@pytest.mark.parametrize("dtype,rows,hidden", [("bf16", 20001, 384), ("bf16", 601, 8192),
                                               ("f32", 3001, 768), ("bf16", 777, 1001)])
def test_low_precision_parameter_gradients(cuda_lib, dtype, rows, hidden, mode, gdt):
    # The down cast after the outer reduction (PR 165370's epilogue): each
    # column total is rounded once to bf16 / fp16. Every value is within one
    # unit of the oracle's total rounded to that type, and equals the fp32
    # result of the same partials rounded to it unless that was a double
    # rounding (the fp64 total lying within an fp32 ulp of a tie).
    from oracle import round_to_format
    from _parity import ulp
    fmt = "bf16" if gdt == torch.bfloat16 else "f16"
    w = wl(dtype, rows, hidden, mode)
    inp = make_inputs(w, seed=13)
    ref = oracle_fwd(w, inp)
    dt = W.TORCH_DTYPES[w.dtype]
    x_sum = torch.from_numpy(ref["sum"]).to(dt)
    mean = None if ref["mean"] is None else torch.from_numpy(ref["mean"]).float()
    rstd = torch.from_numpy(ref["rstd"]).float()
    bref = oracle_bwd_rows(w, inp["dy"], x_sum, inp["gamma"], mean, rstd, slice(None))
    lo = gpu_bwd(cuda_lib, w, inp["dy"], x_sum, inp["gamma"], mean, rstd, need_dbias=True,
                 grad_dtype=gdt)
    hi = gpu_bwd(cuda_lib, w, inp["dy"], x_sum, inp["gamma"], mean, rstd, need_dbias=True)
    assert lo["guards_ok"]
    names = ["dgamma", "dbias"] + (["dbeta"] if mode == W.LAYERNORM else [])
    for k in names:
        got = as_f64(lo[k])
        want = round_to_format(bref[k], fmt)
        # the ulp floor of reading G: a column total that cancels to ~0 is
        # measured on the scale of the vector (2^-8 of its largest entry)
        mag = np.maximum(abs(bref[k]), np.ldexp(abs(bref[k]).max(), -8))
        d = abs(got - want) / ulp(mag, fmt)
        assert d.max() <= 1.0, (k, float(d.max()))
        same = (got == round_to_format(as_f64(hi[k]), fmt)).mean()
        assert same >= 0.999, (k, same)


def test_dbias_on_empty_rows_is_zero(cuda_lib):
    w = wl("bf16", 0, 384, W.LAYERNORM)
    inp = make_inputs(w, seed=12)
    got = gpu_bwd(cuda_lib, w, inp["dy"], inp["x"], inp["gamma"], torch.zeros(0),
                  torch.zeros(0), need_dbias=True)
    assert got["guards_ok"] and (got["dbias"] == 0).all()
