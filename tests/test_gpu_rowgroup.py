"""GPU parity of the backward's row-group kernels: widths whose lane-group
accumulators would not fit in registers run with 64 or 128 threads per row
(LayerNorm from 6 vectors per lane, LayerNorm with dbias from 4). Row counts
leave ragged last tiles (4 or 2 rows per tile)."""

import pytest
import torch

import workloads as W
from _parity import (check_elementwise, check_rel_l2, dx_row_scale, gpu_bwd, oracle_bwd_rows,
                     oracle_fwd)
from workloads import Workload, as_f64, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,rows,hidden,mode,dbias", [
    ("bf16", 1001, 1536, W.LAYERNORM, False),    # 64 threads x 3 vectors
    ("bf16", 1003, 2048, W.LAYERNORM, False),    # 64 x 4
    ("f16", 999, 1280, W.LAYERNORM, True),       # 64 x 3, with dbias
    ("bf16", 1002, 1024, W.LAYERNORM, True),     # 64 x 2, with dbias
    ("f32", 1001, 1024, W.LAYERNORM, True),      # 64 x 4 of 4-element vectors
    ("bf16", 997, 2048, W.RMSNORM, True),        # RMSNorm + dbias: 64 x 4
    ("f16", 515, 1472, W.LAYERNORM, False),      # 184 vectors: 64 x 3 with idle lanes
])
def test_rowgroup_backward_matches_oracle(cuda_lib, dtype, rows, hidden, mode, dbias):
    w = Workload(name="rg", dtype=dtype, rows=rows, hidden=hidden, mode=mode, eps=1e-5,
                 x_std=1.0, residual_std=1.0, bias_std=0.1, gamma_std=0.1,
                 beta_std=0.1 if mode == W.LAYERNORM else None)
    inp = make_inputs(w, seed=21)
    ref = oracle_fwd(w, inp)
    dt = W.TORCH_DTYPES[dtype]
    x_sum = torch.from_numpy(ref["sum"]).to(dt)
    mean = None if ref["mean"] is None else torch.from_numpy(ref["mean"]).float()
    rstd = torch.from_numpy(ref["rstd"]).float()
    bref = oracle_bwd_rows(w, inp["dy"], x_sum, inp["gamma"], mean, rstd, slice(None))
    got = gpu_bwd(cuda_lib, w, inp["dy"], x_sum, inp["gamma"], mean, rstd, need_dbias=dbias)
    assert got["guards_ok"]
    check_elementwise(as_f64(got["dx"]), bref["dx_exact"], dtype, "dx",
                      scale_rows=dx_row_scale(as_f64(inp["dy"]), as_f64(inp["gamma"]),
                                              as_f64(rstd), w.zero_centered_gamma))
    check_rel_l2(as_f64(got["dgamma"]), bref["dgamma"], 1e-4, "dgamma")
    if mode == W.LAYERNORM:
        check_rel_l2(as_f64(got["dbeta"]), bref["dbeta"], 1e-4, "dbeta")
    if dbias:
        check_rel_l2(as_f64(got["dbias"]), bref["dbias"], 1e-4, "dbias")


def test_rowgroup_backward_is_deterministic(cuda_lib):
    w = Workload(name="rg_det", dtype="bf16", rows=4099, hidden=1536, mode=W.LAYERNORM,
                 eps=1e-5, gamma_std=0.1, beta_std=0.1)
    inp = make_inputs(w, seed=22)
    mean = torch.zeros(w.rows)
    rstd = torch.ones(w.rows)
    a = gpu_bwd(cuda_lib, w, inp["dy"], inp["x"], inp["gamma"], mean, rstd)
    b = gpu_bwd(cuda_lib, w, inp["dy"], inp["x"], inp["gamma"], mean, rstd)
    assert torch.equal(a["dgamma"].view(torch.int32), b["dgamma"].view(torch.int32))
    assert torch.equal(a["dbeta"].view(torch.int32), b["dbeta"].view(torch.int32))
    assert torch.equal(a["dx"].view(torch.int16), b["dx"].view(torch.int16))
