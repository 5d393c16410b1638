"""GPU parity on the five workloads of the block, through the C ABI.

Small workloads are compared element by element over every row. The two
large ones (576000 x 384 and 16384 x 8192) run at full size in the same launch
configuration bench.py times; their per-row outputs are compared on a seeded
sample of rows (plus the first and last rows), their column reductions
(dgamma, dbeta) and amax over every row.

The stored sum is held to the plain 2-ulp rule (no row-scale floor: the add
does not cancel below its own rounding). For y and dx the row-scale floor
applies, and the number of elements it decided (more than 2 ulp off by the
plain rule) is recorded with each test (pytest's record_property) and must
stay below 1e-3 of the elements; the rows whose mean the row-scale rule
decided are recorded too.
"""

import numpy as np
import pytest
import torch

import workloads as W
from _parity import (amax_bits_got, dx_row_scale, amax_bits_of, check_elementwise, check_mean, check_rel,
                     check_rel_l2, gpu_bwd, gpu_fwd, oracle_bwd_reductions, oracle_bwd_rows,
                     oracle_fwd, oracle_stats_full, rows_f64)
from workloads import as_f64, make_inputs

pytestmark = pytest.mark.gpu


def sample_rows(R, n, seed=123):
    rng = np.random.default_rng(seed)
    pick = rng.choice(R, size=min(n, R), replace=False)
    edge = np.array([0, 1, R // 2, R - 2, R - 1])
    return np.unique(np.concatenate([pick, edge[edge < R]]))


MAX_FLOORED = 1e-3


def _record(record, rep):
    if record is None:
        return
    for k in ("floored", "floored_frac", "worst_ulp_raw", "within1_raw", "row_scale_decided",
              "row_scale_decided_frac"):
        if k in rep:
            record(f"{rep['what']}_{k}", rep[k])


def check_fwd(w, got, ref, rows=None, record=None):
    sel = (lambda t: rows_f64(t, rows))
    assert got["guards_ok"]
    if "sum" in got:
        _record(record, check_elementwise(sel(got["sum"]), ref["sum"], w.dtype, "sum",
                                          row_scale=False))
    # RMSNorm's y has no cancellation, so it takes the plain rule (no floor).
    _record(record, check_elementwise(sel(got["y"]), ref["y_exact"], w.dtype, "y",
                                      row_scale=w.mode == W.LAYERNORM,
                                      max_floored=MAX_FLOORED))
    check_rel(sel(got["rstd"]), ref["rstd_exact"], 1e-5, "rstd")
    if w.mode == W.LAYERNORM:
        _record(record, check_mean(sel(got["mean"]), ref["mean_exact"], ref["sum"]))
    if "amax" in got:
        # bit-exact against the kernel's own stored y ...
        assert amax_bits_got(got["amax"]) == amax_bits_of(got["y"])
        if rows is None:
            # ... and within 2 ulp of the oracle's amax, like any element of y
            check_elementwise(np.array([float(got["amax"][0])]), np.array([ref["amax"]]),
                              w.dtype, "amax")


def check_bwd(w, got, ref_rows, dg_ref, db_ref, dy, gamma, rstd, rows=None, record=None):
    assert got["guards_ok"]
    dx = rows_f64(got["dx"], rows)
    scale = dx_row_scale(rows_f64(dy, rows), rows_f64(gamma), rows_f64(rstd, rows),
                         w.zero_centered_gamma)
    _record(record, check_elementwise(dx, ref_rows["dx_exact"], w.dtype, "dx", scale_rows=scale,
                                      max_floored=MAX_FLOORED))
    check_rel_l2(as_f64(got["dgamma"]), dg_ref, 1e-4, "dgamma")
    if db_ref is not None:
        check_rel_l2(as_f64(got["dbeta"]), db_ref, 1e-4, "dbeta")


def run_fwd_bwd_small(lib, w, record=None):
    """Full-tensor forward parity, then backward parity with the backward fed
    the oracle's forward outputs, then the GPU forward -> GPU backward chain."""
    inp = make_inputs(w, seed=0)
    ref = oracle_fwd(w, inp)
    got = gpu_fwd(lib, w, inp)
    check_fwd(w, got, ref, record=record)
    if not w.backward:
        return
    dt = W.TORCH_DTYPES[w.dtype]
    x_sum = torch.from_numpy(ref["sum"]).to(dt)
    mean = None if ref["mean"] is None else torch.from_numpy(ref["mean"]).float()
    rstd = torch.from_numpy(ref["rstd"]).float()
    bref = oracle_bwd_rows(w, inp["dy"], x_sum, inp["gamma"], mean, rstd, slice(None))
    bgot = gpu_bwd(lib, w, inp["dy"], x_sum, inp["gamma"], mean, rstd)
    check_bwd(w, bgot, bref, bref["dgamma"], bref["dbeta"], inp["dy"], inp["gamma"], rstd,
              record=record)
    # chain: the backward consumes the GPU forward's own outputs
    cgot = gpu_bwd(lib, w, inp["dy"], got["sum"], inp["gamma"], got.get("mean"), got["rstd"])
    check_bwd(w, cgot, bref, bref["dgamma"], bref["dbeta"], inp["dy"], inp["gamma"], rstd)


def test_layernorm_fp32_4096x384(cuda_lib, record_property):
    run_fwd_bwd_small(cuda_lib, W.LN_F32_4096x384, record_property)


def test_fwd_bias_residual_zero_centered_amax_bf16_32768x768(cuda_lib, record_property):
    run_fwd_bwd_small(cuda_lib, W.FWD_AMAX_BF16_32768x768, record_property)


@pytest.mark.parametrize("hidden", [320, 640, 1280])
def test_unet_layernorm_fp16_8192(cuda_lib, hidden, record_property):
    run_fwd_bwd_small(cuda_lib, W.UNET_F16[hidden], record_property)


@pytest.mark.parametrize("w", [W.BWD_BF16_576000x384_LN, W.BWD_BF16_576000x384_RMS],
                         ids=lambda w: w.name)
def test_backward_bf16_576000x384(cuda_lib, w, record_property):
    """Backward only; mean/rstd come from the oracle's fp64 forward of x."""
    inp = make_inputs(w, seed=0)
    mean, rstd = oracle_stats_full(w, inp["x"])
    got = gpu_bwd(cuda_lib, w, inp["dy"], inp["x"], inp["gamma"], mean, rstd)
    rows = sample_rows(w.rows, 20000)
    ref_rows = oracle_bwd_rows(w, inp["dy"], inp["x"], inp["gamma"], mean, rstd, rows)
    dg, db = oracle_bwd_reductions(w, inp["dy"], inp["x"], inp["gamma"], mean, rstd)
    check_bwd(w, got, ref_rows, dg, db, inp["dy"], inp["gamma"], rstd, rows=rows,
              record=record_property)


def run_large_fwd_bwd(lib, w, record=None):
    inp = make_inputs(w, seed=0)
    got = gpu_fwd(lib, w, inp)
    rows = sample_rows(w.rows, 4000 if w.hidden > 4096 else 20000)
    ref = oracle_fwd(w, inp, rows=rows)
    check_fwd(w, got, ref, rows=rows, record=record)
    # amax over the whole tensor: bit-exact against the kernel's stored y.
    if w.amax:
        assert amax_bits_got(got["amax"]) == amax_bits_of(got["y"])
    # The backward is fed the oracle's forward outputs for every row (stored
    # sum and fp32 statistics), so no oracle input comes from the GPU.
    dt = W.TORCH_DTYPES[w.dtype]
    full = oracle_fwd_stats_and_sum(w, inp)
    x_sum = full["sum"]
    mean, rstd = full["mean"], full["rstd"]
    bgot = gpu_bwd(lib, w, inp["dy"], x_sum, inp["gamma"], mean, rstd)
    ref_rows = oracle_bwd_rows(w, inp["dy"], x_sum, inp["gamma"], mean, rstd, rows)
    dg, db = oracle_bwd_reductions(w, inp["dy"], x_sum, inp["gamma"], mean, rstd)
    check_bwd(w, bgot, ref_rows, dg, db, inp["dy"], inp["gamma"], rstd, rows=rows,
              record=record)
    assert bgot["dx"].dtype == dt


def oracle_fwd_stats_and_sum(w, inp, chunk=16384):
    """The oracle forward over every row, keeping the stored sum and the fp32
    statistics (as torch tensors) for the backward."""
    R, H = w.rows, w.hidden
    dt = W.TORCH_DTYPES[w.dtype]
    x_sum = torch.empty(R, H, dtype=dt)
    rstd = torch.empty(R, dtype=torch.float32)
    mean = torch.empty(R, dtype=torch.float32) if w.mode == W.LAYERNORM else None
    for i in range(0, R, chunk):
        sl = slice(i, min(R, i + chunk))
        o = oracle_fwd(w, inp, rows=sl)
        x_sum[sl] = torch.from_numpy(o["sum"]).to(dt)
        rstd[sl] = torch.from_numpy(o["rstd"]).float()
        if mean is not None:
            mean[sl] = torch.from_numpy(o["mean"]).float()
    return {"sum": x_sum, "mean": mean, "rstd": rstd}


def test_rmsnorm_bf16_16384x8192_outliers(cuda_lib, record_property):
    run_large_fwd_bwd(cuda_lib, W.RMS_BF16_16384x8192, record_property)


def test_bench_workload_ln_bf16_576000x384(cuda_lib, record_property):
    """The step bench.py times (bias + residual + amax forward, backward)."""
    run_large_fwd_bwd(cuda_lib, W.BENCH_LN_BF16_576000x384, record_property)
