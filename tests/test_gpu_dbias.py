"""GPU parity of the bias gradient (ln_bwd_ex): dbias = sum over rows of dx,
the third column reduction fused into the backward's persistent kernel.

Checked against the oracle's dbias (fp32 rules: relative L2 <= 1e-4), and
dx must be bitwise that of ln_bwd on the same inputs (dgamma/dbeta may differ
in the last bits: the dbias kernel can run a different number of CTAs per SM,
hence a different row partition of the partial sums).
"""

import pytest
import torch

import workloads as W
from _parity import check_rel_l2, gpu_bwd, oracle_bwd_rows, oracle_fwd
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
    plain = gpu_bwd(cuda_lib, w, inp["dy"], x_sum, inp["gamma"], mean, rstd)
    assert ex["guards_ok"]
    check_rel_l2(as_f64(ex["dbias"]), bref["dbias"], 1e-4, "dbias")
    bits = torch.int16 if ex["dx"].element_size() == 2 else torch.int32
    assert torch.equal(ex["dx"].view(bits), plain["dx"].view(bits))
    check_rel_l2(as_f64(ex["dgamma"]), bref["dgamma"], 1e-4, "dgamma")
    if mode == W.LAYERNORM:
        check_rel_l2(as_f64(ex["dbeta"]), bref["dbeta"], 1e-4, "dbeta")


def test_dbias_on_empty_rows_is_zero(cuda_lib):
    w = wl("bf16", 0, 384, W.LAYERNORM)
    inp = make_inputs(w, seed=12)
    got = gpu_bwd(cuda_lib, w, inp["dy"], inp["x"], inp["gamma"], torch.zeros(0),
                  torch.zeros(0), need_dbias=True)
    assert got["guards_ok"] and (got["dbias"] == 0).all()
