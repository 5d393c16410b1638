"""GPU parity of the row softmax (ln_softmax_fwd) against the fp64 oracle.

Tolerances:
* bf16/fp16 output: every element within 2 ulp of the oracle's exact value
  rounded to the dtype, >= 99.9 % within 1 ulp (softmax values are positive
  and do not cancel, so no row-scale floor is needed).
* fp32 output: relative error <= (64 + 2 |x_j - m|) * 2^-24 per element. The
  kernel takes e_j = exp2f(fma(x_j, log2e, -m log2e)): the fma rounds the
  exponent with relative error 2^-24, i.e. an error of |x_j - m| * 2^-24 in
  e_j, and log2e rounded to fp32 adds at most |x_j - m| * 2^-25 (the rounding
  of m log2e is common to the row and cancels in e_j / s); exp2f is within
  2 ulp (2^-22); the fp32 row sum of up to 32 terms per thread, a 5-level
  butterfly and 8 warp partials adds at most ~45 * 2^-24; the warp rescaling
  of the CTA-per-row kernel, the reciprocal and the products a few 2^-24.
* masked (-inf) entries of a finite row are exactly 0; fully masked rows
  (and only those) are NaN in every column.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import round_to_format, softmax_fwd
from workloads import (SMX_BF16_16384x8192, SMX_BF16_576000x384, SMX_F16_8192x1280_MASKED,
                       SMX_F32_4096x384, SoftmaxWorkload, TORCH_DTYPES, as_f64,
                       make_softmax_inputs)
from _parity import Guarded, check_elementwise

pytestmark = pytest.mark.gpu


def run_gpu(lib, x_cpu, *, inplace=False, offset_elems=0):
    """ln_softmax_fwd on a copy of x; returns the CPU result and guard status."""
    R, H = x_cpu.shape
    if inplace:
        g = Guarded((R * H + offset_elems,), x_cpu.dtype)
        y = g.t[offset_elems:].view(R, H)
        y.copy_(x_cpu.to("cuda"))
        lib.ln_softmax_fwd(y, y)
    else:
        xd = torch.empty(R * H + offset_elems, dtype=x_cpu.dtype, device="cuda")
        x = xd[offset_elems:].view(R, H)
        x.copy_(x_cpu.to("cuda"))
        g = Guarded((R * H + offset_elems,), x_cpu.dtype)
        y = g.t[offset_elems:].view(R, H)
        lib.ln_softmax_fwd(x, y)
    torch.cuda.synchronize()
    assert lib.ln_device_error() == 0, "a kernel reported a failed wait"
    return y.cpu(), g.guards_intact()


def check(got, x64, fmt, what):
    ref = softmax_fwd(x64, "f64")
    y = ref["y_exact"]
    got = as_f64(got)
    full_mask = np.isneginf(x64).all(axis=1) if x64.shape[1] else np.zeros(x64.shape[0], bool)
    assert np.isnan(got[full_mask]).all(), f"{what}: fully masked rows must be NaN"
    got, y, xr, m = got[~full_mask], y[~full_mask], x64[~full_mask], ref["max"][~full_mask]
    masked = np.isneginf(xr)
    assert (got[masked] == 0).all(), f"{what}: masked entries must be exactly 0"
    if fmt == "f32":
        assert np.isfinite(got).all(), f"{what}: non-finite output"
        t = np.where(masked, 0.0, np.abs(xr - m[:, None]))
        tol = (64.0 + 2.0 * t) * 2.0 ** -24 * y + 2.0 ** -149
        err = np.abs(got - y)
        worst = float((err / np.maximum(tol, 1e-300)).max()) if err.size else 0.0
        assert (err <= tol).all(), f"{what}: error up to {worst:.2f} x the bound"
        return {"what": what, "worst_of_bound": worst}
    return check_elementwise(got, y, fmt, what, row_scale=False)


# (dtype, rows, hidden): lane groups of 8/16/32 with every N, the CTA-per-row
# kernel at several CTA sizes, ragged last tiles, widths the vector path
# cannot take (scalar kernel) and the largest widths of each path.
SHAPES = [
    ("f32", 4096, 384), ("f32", 257, 4), ("f32", 1000, 40), ("f32", 333, 1000),
    ("f32", 37, 8192), ("f32", 50, 1025), ("f32", 9, 1),
    ("bf16", 1000, 384), ("bf16", 515, 8), ("bf16", 300, 24), ("bf16", 129, 2048),
    ("bf16", 77, 4096), ("bf16", 33, 16384), ("bf16", 100, 1000), ("bf16", 40, 8191),
    ("bf16", 41, 8192), ("bf16", 23, 6144),    # two rows per CTA with an odd row count
    ("bf16", 515, 256), ("bf16", 129, 1536),   # 8 lanes x 4; a 64-thread CTA
    ("bf16", 37, 2560), ("bf16", 31, 3072),    # row-fitted CTAs: 64 x 5, 96 x 4
    ("bf16", 17, 3),
    ("f16", 8192, 320), ("f16", 999, 640), ("f16", 601, 1280), ("f16", 65, 12288),
    ("f16", 31, 7),
]


@pytest.mark.parametrize("dt,R,H", SHAPES)
def test_softmax_matches_oracle(cuda_lib, dt, R, H):
    w = SoftmaxWorkload(name="t", dtype=dt, rows=R, hidden=H, x_std=3.0)
    x = make_softmax_inputs(w, seed=R + H)
    got, guards = run_gpu(cuda_lib, x)
    assert guards
    check(got, as_f64(x), dt, f"{dt} {R}x{H}")


@pytest.mark.parametrize("w", [SMX_F32_4096x384, SMX_F16_8192x1280_MASKED],
                         ids=lambda w: w.name)
def test_softmax_workloads(cuda_lib, w):
    x = make_softmax_inputs(w)
    got, guards = run_gpu(cuda_lib, x)
    assert guards
    check(got, as_f64(x), w.dtype, w.name)


@pytest.mark.parametrize("dt,H", [("bf16", 384), ("f16", 1280), ("f32", 333), ("bf16", 8192)])
def test_softmax_masked_rows(cuda_lib, dt, H):
    w = SoftmaxWorkload(name="m", dtype=dt, rows=203, hidden=H, mask_frac=0.5, masked_rows=5)
    x = make_softmax_inputs(w, seed=7)
    got, _ = run_gpu(cuda_lib, x)
    check(got, as_f64(x), dt, f"masked {dt} {H}")


@pytest.mark.parametrize("dt,H", [("bf16", 384), ("f32", 8192), ("f16", 77)])
def test_softmax_large_logits_need_the_max_shift(cuda_lib, dt, H):
    # exp of these values overflows fp32; only the max subtraction keeps y finite.
    w = SoftmaxWorkload(name="big", dtype=dt, rows=64, hidden=H, x_std=1.0)
    x = make_softmax_inputs(w, seed=3)
    x = (x.to(torch.float32) + 200.0).to(x.dtype)
    got, _ = run_gpu(cuda_lib, x)
    check(got, as_f64(x), dt, f"big {dt}")


@pytest.mark.parametrize("dt,H", [("bf16", 384), ("bf16", 4096), ("f32", 100), ("f16", 1000)])
def test_softmax_in_place(cuda_lib, dt, H):
    w = SoftmaxWorkload(name="ip", dtype=dt, rows=211, hidden=H)
    x = make_softmax_inputs(w, seed=11)
    got, guards = run_gpu(cuda_lib, x, inplace=True)
    assert guards
    check(got, as_f64(x), dt, f"in place {dt} {H}")


@pytest.mark.parametrize("dt,H", [("bf16", 384), ("f32", 256)])
def test_softmax_unaligned_pointers_take_the_scalar_path(cuda_lib, dt, H):
    w = SoftmaxWorkload(name="ua", dtype=dt, rows=123, hidden=H)
    x = make_softmax_inputs(w, seed=13)
    got, guards = run_gpu(cuda_lib, x, offset_elems=1)
    assert guards
    check(got, as_f64(x), dt, f"unaligned {dt} {H}")


def test_softmax_zero_rows_is_a_no_op(cuda_lib):
    x = torch.empty(0, 384, dtype=torch.bfloat16, device="cuda")
    cuda_lib.ln_softmax_fwd(x, torch.empty_like(x))
    torch.cuda.synchronize()


def test_softmax_rows_are_independent_of_their_neighbours(cuda_lib):
    # A row's result does not depend on the tile or CTA it lands in: the
    # same row computed alone and inside a large batch is bitwise equal.
    w = SoftmaxWorkload(name="ind", dtype="bf16", rows=5000, hidden=384)
    x = make_softmax_inputs(w, seed=17)
    big, _ = run_gpu(cuda_lib, x)
    for r in (0, 1, 2500, 4999):
        one, _ = run_gpu(cuda_lib, x[r:r + 1].contiguous())
        assert torch.equal(one[0].view(torch.int16), big[r].view(torch.int16))


@pytest.mark.parametrize("w", [SMX_BF16_576000x384, SMX_BF16_16384x8192], ids=lambda w: w.name)
def test_softmax_full_size_sampled_rows(cuda_lib, w):
    # The full workload in the launch configuration the benchmark times;
    # the oracle checks a sample of rows (spread over the grid, the first
    # and last tiles) and every row must sum to 1 within the rounding of y.
    x = make_softmax_inputs(w)
    xd = x.to("cuda")
    y = torch.empty_like(xd)
    cuda_lib.ln_softmax_fwd(xd, y)
    torch.cuda.synchronize()
    assert cuda_lib.ln_device_error() == 0
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.arange(16), np.arange(w.rows - 16, w.rows),
                                     rng.integers(0, w.rows, 2000)]))
    idx = torch.as_tensor(rows, dtype=torch.long, device="cuda")
    got = y.index_select(0, idx).cpu()
    check(got, as_f64(x[torch.as_tensor(rows)]), w.dtype, w.name)
    sums = y.to(torch.float64).sum(dim=1)
    # each of H outputs carries at most half an ulp of rounding (2^-9 relative for bf16)
    assert float((sums - 1).abs().max()) <= 2.0 ** -8
