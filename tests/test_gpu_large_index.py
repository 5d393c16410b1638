"""Tensors of more than 2^31 elements (more than 4 GiB of bf16).

Every row offset in the kernels is 64-bit; these tests hold the library to
that on shapes where a 32-bit element or byte offset would wrap. Each input
is a seeded block of rows tiled many times over on the device, so the full
tensor passes 2^31 elements while the oracle only has to see the block:

* every row-wise output (y, the stored sum, mean, rstd, dx, the softmax) of
  row r must be bit-identical to that of row r mod block, checked over every
  row on the device (one kernel computes every row the same way, so a row
  read or written through a wrapped offset shows up as a mismatch);
* the block's rows are compared with the fp64 oracle under the parity
  tests' tolerances;
* dgamma and dbeta are sums over rows, so they equal reps times the block's
  (relative L2 error <= 1e-4); amax equals the block's, bit for bit.

Each test holds about 28 GB of device memory and frees it when done.
"""

import gc

import numpy as np
import pytest
import torch

import workloads as W
from _parity import (amax_bits_of, check_elementwise, check_mean, check_rel, check_rel_l2,
                     dx_row_scale, oracle_bwd_rows, oracle_fwd)
from oracle import norm_fwd_from_partials, row_tile_partials, softmax_fwd
from workloads import TORCH_DTYPES, Workload, as_f64, make_inputs

pytestmark = pytest.mark.gpu

TWO31 = 2 ** 31


@pytest.fixture(autouse=True)
def _free_device_memory():
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _tile(t, reps):
    """A CPU [block, ...] tensor tiled reps times along rows on the device."""
    if t is None:
        return None
    d = t.to("cuda")
    return d.repeat(reps, *([1] * (d.dim() - 1))).contiguous()


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def assert_rows_repeat(t, block, what):
    """Row r of t equals row r mod block, bit for bit, over every row."""
    R = t.shape[0]
    assert R % block == 0
    v = _bits(t).view(R // block, block, *t.shape[1:])
    first = v[:1]
    step = max(1, (1 << 28) // max(1, v[0].numel()))
    for i in range(0, v.shape[0], step):
        chunk = v[i:i + step]
        same = (chunk == first).reshape(chunk.shape[0], -1).all(dim=1)
        if not bool(same.all()):
            bad = i + int(torch.nonzero(~same)[0, 0])
            raise AssertionError(f"{what}: copy {bad} of the block (rows from {bad * block}) "
                                 "differs from the first")


def _fwd_bwd(lib, w, reps):
    """Forward then backward over the tiled block; returns device outputs."""
    inp = make_inputs(w, seed=77)
    dt = TORCH_DTYPES[w.dtype]
    R, H = w.rows * reps, w.hidden
    assert R * H > TWO31
    rms = w.mode == W.RMSNORM
    x, res, dy = _tile(inp["x"], reps), _tile(inp["residual"], reps), _tile(inp["dy"], reps)
    gamma = inp["gamma"].to("cuda")
    beta = inp["beta"].to("cuda") if inp["beta"] is not None else None
    bias = inp["bias"].to("cuda") if inp["bias"] is not None else None
    out = {"y": torch.empty(R, H, dtype=dt, device="cuda"),
           "sum": torch.empty(R, H, dtype=dt, device="cuda") if res is not None else None,
           "rstd": torch.empty(R, dtype=torch.float32, device="cuda"),
           "mean": None if rms else torch.empty(R, dtype=torch.float32, device="cuda"),
           "amax": torch.empty(1, dtype=torch.float32, device="cuda")}
    lib.ln_fwd(x, bias, res, gamma, beta, w.eps, w.mode, w.zero_centered_gamma, out["sum"],
               out["y"], out["mean"], out["rstd"], out["amax"])
    del res
    x_sum = out["sum"] if out["sum"] is not None else x
    out["dx"] = torch.empty(R, H, dtype=dt, device="cuda")
    out["dgamma"] = torch.empty(H, dtype=torch.float32, device="cuda")
    out["dbeta"] = None if rms else torch.empty(H, dtype=torch.float32, device="cuda")
    lib.ln_bwd(dy, x_sum, gamma, out["mean"], out["rstd"], out["dx"], out["dgamma"],
               out["dbeta"], mode=w.mode, zero_centered_gamma=w.zero_centered_gamma)
    torch.cuda.synchronize()
    assert lib.ln_device_error() == 0, "a kernel reported a failed wait"
    del x, dy
    return inp, out


# 6,000,000 x 384 (2.30e9 elements): lane-group forward and backward kernels.
# 270,000 x 8192 (2.21e9 elements): CTA-per-row forward, prefetching backward.
CASES = [
    (Workload(name="ln_bf16_4800x384_bias_res", dtype="bf16", rows=4800, hidden=384,
              mode=W.LAYERNORM, eps=1e-5, residual_std=1.0, bias_std=0.1, gamma_std=0.1,
              beta_std=0.1, amax=True), 1250),
    (Workload(name="rms_bf16_1000x8192_res", dtype="bf16", rows=1000, hidden=8192,
              mode=W.RMSNORM, eps=1e-6, residual_std=1.0, gamma_std=0.1, amax=True), 270),
]


@pytest.mark.parametrize("w,reps", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_fwd_bwd_past_2_31_elements(cuda_lib, w, reps):
    inp, out = _fwd_bwd(cuda_lib, w, reps)
    B = w.rows
    for k in ("y", "sum", "mean", "rstd", "dx"):
        if out[k] is not None:
            assert_rows_repeat(out[k], B, k)
    blk = {k: (v[:B].cpu() if v is not None and v.dim() and v.shape[0] == B * reps else None)
           for k, v in out.items()}
    ref = oracle_fwd(w, inp)
    if blk["sum"] is not None:
        check_elementwise(as_f64(blk["sum"]), ref["sum"], w.dtype, "sum", row_scale=False)
    check_elementwise(as_f64(blk["y"]), ref["y_exact"], w.dtype, "y",
                      row_scale=w.mode == W.LAYERNORM, max_floored=1e-3)
    check_rel(as_f64(blk["rstd"]), ref["rstd_exact"], 1e-5, "rstd")
    if w.mode == W.LAYERNORM:
        check_mean(as_f64(blk["mean"]), ref["mean_exact"], ref["sum"])
    amax = out["amax"].cpu()
    assert int(amax.numpy().view(np.uint32)[0]) == amax_bits_of(blk["y"])

    # The oracle's backward on the block, fed the oracle's forward outputs.
    dt = TORCH_DTYPES[w.dtype]
    x_sum = torch.from_numpy(ref["sum"]).to(dt)
    mean = None if ref["mean"] is None else torch.from_numpy(ref["mean"]).float()
    rstd = torch.from_numpy(ref["rstd"]).float()
    bref = oracle_bwd_rows(w, inp["dy"], x_sum, inp["gamma"], mean, rstd, slice(None))
    scale = dx_row_scale(as_f64(inp["dy"]), as_f64(inp["gamma"]), as_f64(rstd),
                         w.zero_centered_gamma)
    check_elementwise(as_f64(blk["dx"]), bref["dx_exact"], w.dtype, "dx", scale_rows=scale,
                      max_floored=1e-3)
    check_rel_l2(as_f64(out["dgamma"].cpu()), reps * bref["dgamma"], 1e-4, "dgamma")
    if w.mode == W.LAYERNORM:
        check_rel_l2(as_f64(out["dbeta"].cpu()), reps * bref["dbeta"], 1e-4, "dbeta")


def test_softmax_past_2_31_elements(cuda_lib):
    B, H, reps = 4800, 384, 1250
    rng = np.random.Generator(np.random.PCG64(78))
    xb = torch.from_numpy(3.0 * rng.standard_normal((B, H))).to(torch.bfloat16)
    x = _tile(xb, reps)
    assert x.numel() > TWO31
    y = torch.empty_like(x)
    cuda_lib.ln_softmax_fwd(x, y)
    torch.cuda.synchronize()
    assert cuda_lib.ln_device_error() == 0
    del x
    assert_rows_repeat(y, B, "softmax y")
    ref = softmax_fwd(as_f64(xb), "f64")
    check_elementwise(as_f64(y[:B].cpu()), ref["y_exact"], "bf16", "softmax y", row_scale=False)


def test_fwd_from_partials_past_2_31_elements(cuda_lib):
    w = Workload(name="p_bf16_4800x384", dtype="bf16", rows=4800, hidden=384,
                 mode=W.LAYERNORM, eps=1e-5, gamma_std=0.05, beta_std=0.05, backward=False)
    reps, tile = 1250, 128
    inp = make_inputs(w, seed=79)
    x64 = as_f64(inp["x"])
    psum, psq = row_tile_partials(x64, tile, "sum_sq", fmt="f32")
    ps = _tile(torch.from_numpy(psum.astype(np.float32)), reps)
    pq = _tile(torch.from_numpy(psq.astype(np.float32)), reps)
    x = _tile(inp["x"], reps)
    R, H = x.shape
    assert R * H > TWO31
    y = torch.empty_like(x)
    mean = torch.empty(R, dtype=torch.float32, device="cuda")
    rstd = torch.empty(R, dtype=torch.float32, device="cuda")
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    cuda_lib.ln_fwd_from_partials(x, ps, pq, tile, "sum_sq", inp["gamma"].to("cuda"),
                                  inp["beta"].to("cuda"), w.eps, w.mode, False, y, mean, rstd,
                                  amax)
    torch.cuda.synchronize()
    assert cuda_lib.ln_device_error() == 0
    del x, ps, pq
    for t, k in ((y, "y"), (mean, "mean"), (rstd, "rstd")):
        assert_rows_repeat(t, w.rows, k)
    ref = norm_fwd_from_partials(x64, psum, psq, tile, "sum_sq", as_f64(inp["gamma"]),
                                 as_f64(inp["beta"]), w.eps, w.mode, False, w.dtype)
    yb = y[:w.rows].cpu()
    check_elementwise(as_f64(yb), ref["y_exact"], w.dtype, "y", max_floored=1e-3)
    check_rel(as_f64(rstd[:w.rows].cpu()), ref["rstd_exact"], 1e-5, "rstd")
    check_mean(as_f64(mean[:w.rows].cpu()), ref["mean_exact"], x64)
    assert int(amax.cpu().numpy().view(np.uint32)[0]) == amax_bits_of(yb)
