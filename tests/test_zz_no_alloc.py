"""ln_bwd_noalloc, the backward for callers that cannot allocate device memory.

Some callers must not call cudaMalloc (or any allocator) around a backward
pass: a framework that owns all device memory through its own caching pool,
a runtime whose memory budget is fixed up front, or a hot path where an
allocation (which may synchronise the device) is not allowed. For them the
library keeps the backward's scratch (the per-CTA dgamma/dbeta partials) in a
static device array instead of a caller workspace.

These tests call that entry point through the C ABI twice in a row on the
same inputs and check both results against the fp64 oracle (dx element by
element, dgamma/dbeta over every row) with the parity tests' tolerances, and
against ln_bwd with a caller workspace (the same kernels and partial order,
so the same bits). They also check the size limit, on both sides of it.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""

import pytest
import torch

import workloads as W
from _parity import (check_elementwise, check_rel_l2, dx_row_scale, oracle_bwd_reductions,
                     oracle_bwd_rows, oracle_fwd)
from workloads import as_f64, make_inputs

pytestmark = pytest.mark.gpu


def _oracle_forward(w, seed):
    """Inputs and the oracle's forward outputs (stored sum, fp32 statistics),
    so no input of the backward comes from the CUDA path."""
    inp = make_inputs(w, seed=seed)
    ref = oracle_fwd(w, inp)
    dt = W.TORCH_DTYPES[w.dtype]
    x_sum = torch.from_numpy(ref["sum"]).to(dt)
    mean = None if ref["mean"] is None else torch.from_numpy(ref["mean"]).float()
    rstd = torch.from_numpy(ref["rstd"]).float()
    return inp, x_sum, mean, rstd


def _run_twice_and_check(nf, w, seed=7):
    dev = torch.device("cuda")
    inp, x_sum, mean, rstd = _oracle_forward(w, seed)
    rms = w.mode == W.RMSNORM
    H = w.hidden
    g = {"dy": inp["dy"].to(dev), "sum": x_sum.to(dev), "gamma": inp["gamma"].to(dev),
         "mean": None if rms else mean.to(dev), "rstd": rstd.to(dev)}

    def outputs():
        return (torch.full_like(g["dy"], float("nan")),
                torch.full((H,), float("nan"), device=dev),
                None if rms else torch.full((H,), float("nan"), device=dev))

    ref_rows = oracle_bwd_rows(w, inp["dy"], x_sum, inp["gamma"], mean, rstd, slice(None))
    dg_ref, db_ref = oracle_bwd_reductions(w, inp["dy"], x_sum, inp["gamma"], mean, rstd)
    scale = dx_row_scale(as_f64(inp["dy"]), as_f64(inp["gamma"]), as_f64(rstd),
                         w.zero_centered_gamma)

    dx_ws, dg_ws, db_ws = outputs()
    nf.ln_bwd(g["dy"], g["sum"], g["gamma"], g["mean"], g["rstd"], dx_ws, dg_ws, db_ws,
              mode=w.mode, zero_centered_gamma=w.zero_centered_gamma)
    for _ in range(2):
        dx, dg, db = outputs()
        nf.ln_bwd_noalloc(g["dy"], g["sum"], g["gamma"], g["mean"], g["rstd"], dx, dg, db,
                          mode=w.mode, zero_centered_gamma=w.zero_centered_gamma)
        torch.cuda.synchronize()
        assert nf.ln_device_error() == 0
        # against the oracle
        check_elementwise(as_f64(dx.cpu()), ref_rows["dx_exact"], w.dtype, "dx",
                          scale_rows=scale)
        check_rel_l2(as_f64(dg.cpu()), dg_ref, 1e-4, "dgamma")
        if not rms:
            check_rel_l2(as_f64(db.cpu()), db_ref, 1e-4, "dbeta")
        # against the workspace backward: the same kernels, partials and order
        assert torch.equal(dx, dx_ws)
        assert torch.equal(dg, dg_ws)
        if not rms:
            assert torch.equal(db, db_ws)


@pytest.mark.parametrize("w", [
    W.BENCH_LN_BF16_576000x384.with_(rows=50001),
    W.RMS_BF16_16384x8192.with_(rows=1500, outlier_frac=0.0),
    W.LN_F32_4096x384,
    W.FWD_AMAX_BF16_32768x768.with_(rows=3001, backward=True),   # zero-centered gamma
], ids=lambda w: w.name)
def test_noalloc_backward_matches_oracle_twice(cuda_lib, w):
    _run_twice_and_check(cuda_lib, w)


def test_noalloc_backward_just_under_the_limit(cuda_lib):
    """The widest bf16 LayerNorm the array holds, found from the entry
    point's own answers (LN_OK up to it, LN_ERR_SCRATCH_LIMIT past it; a
    refused call enqueues nothing), runs and matches the oracle twice."""
    nf = cuda_lib
    lib = nf.load_library()
    rows, h_max = 400, 16384
    dev = "cuda"
    z = lambda n, dt: torch.zeros(n, dtype=dt, device=dev)
    dy, xs, dx = (z(rows * h_max, torch.bfloat16) for _ in range(3))
    gm = z(h_max, torch.bfloat16)
    mean, rstd = z(rows, torch.float32), z(rows, torch.float32)
    dg, db = z(h_max, torch.float32), z(h_max, torch.float32)

    def status(H):
        return lib.ln_bwd_noalloc(dy.data_ptr(), xs.data_ptr(), gm.data_ptr(), mean.data_ptr(),
                                  rstd.data_ptr(), dx.data_ptr(), dg.data_ptr(), db.data_ptr(),
                                  None, rows, H, nf.LN_BF16, nf.LN_LAYERNORM, 0)

    lo, hi = 8, h_max          # status(lo) is OK, status(hi) is the limit
    assert status(lo) == nf.LN_OK
    assert status(hi) == nf.LN_ERR_SCRATCH_LIMIT
    while hi - lo > 8:
        mid = (lo + hi) // 16 * 8
        st = status(mid)
        assert st in (nf.LN_OK, nf.LN_ERR_SCRATCH_LIMIT), nf.ln_status_string(st)
        if st == nf.LN_OK:
            lo = mid
        else:
            hi = mid
    torch.cuda.synchronize()
    assert nf.ln_device_error() == 0
    H = lo
    # Rows this wide keep one partial row (dgamma and dbeta, fp32) per SM,
    # so the limit sits where SMs x 2 x H x 4 bytes reach the array's size.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert H >= 0.99 * nf.LN_NOALLOC_SCRATCH_BYTES / (sms * 2 * 4) - 8, (H, sms)
    w = W.BENCH_LN_BF16_576000x384.with_(rows=rows, hidden=H, name=f"noalloc_ln_bf16_{rows}x{H}")
    _run_twice_and_check(nf, w, seed=8)


def test_noalloc_backward_reports_scratch_limit(cuda_lib):
    # LayerNorm at hidden 16384 keeps one partial row per SM: 152 SMs x 2 x
    # 16384 x 4 bytes of partials, past the array.
    nf = cuda_lib
    lib = nf.load_library()
    rows, H = 400, 16384
    need = nf.ln_bwd_workspace_bytes(rows, H, torch.bfloat16, "layernorm")
    assert need > nf.LN_NOALLOC_SCRATCH_BYTES
    dev = "cuda"
    t = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt, device=dev)
    dy, xs, gm, dx = t(rows, H), t(rows, H), t(H), t(rows, H)
    mean, rstd = t(rows, dt=torch.float32), t(rows, dt=torch.float32)
    dg, db = t(H, dt=torch.float32), t(H, dt=torch.float32)
    st = lib.ln_bwd_noalloc(dy.data_ptr(), xs.data_ptr(), gm.data_ptr(), mean.data_ptr(),
                            rstd.data_ptr(), dx.data_ptr(), dg.data_ptr(), db.data_ptr(),
                            None, rows, H, nf.LN_BF16, nf.LN_LAYERNORM, 0)
    assert st == nf.LN_ERR_SCRATCH_LIMIT, nf.ln_status_string(st)
    assert "SCRATCH_LIMIT" in nf.ln_status_string(st)
    # nothing was enqueued: dx is untouched
    torch.cuda.synchronize()
    assert not dx.any()
