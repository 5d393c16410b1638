"""ln_bwd_noalloc, the backward for callers that cannot allocate device memory.

Some callers must not call cudaMalloc (or any allocator) around a backward
pass: code captured into a CUDA graph or driven by a framework that owns all
device memory through its own pool, and runtimes with a fixed memory budget
set up front. For them the library keeps the backward's scratch (the per-CTA
dgamma/dbeta partials) in a static device array instead of a caller
workspace. This test calls that entry point through the C ABI twice in a row
and checks both results against ln_bwd with a caller workspace, with the
tolerances of the parity tests; it also checks the size limit is reported.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""

import ctypes

import pytest
import torch

import workloads as W
from _parity import check_elementwise, check_rel_l2, dx_row_scale
from workloads import as_f64, make_inputs

pytestmark = pytest.mark.gpu


def _forward(nf, w, dev):
    inp = make_inputs(w, seed=7)
    g = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    f = nf.fused_norm_fwd(g["x"], g["gamma"], g["beta"], bias=g["bias"], residual=g["residual"],
                          eps=w.eps, mode=w.mode, store_sum=True)
    return g, f


@pytest.mark.parametrize("w", [
    W.BENCH_LN_BF16_576000x384.with_(rows=50001),
    W.RMS_BF16_16384x8192.with_(rows=1500, outlier_frac=0.0),
    W.LN_F32_4096x384,
], ids=lambda w: w.name)
def test_noalloc_backward_matches_workspace_backward(cuda_lib, w):
    nf = cuda_lib
    dev = torch.device("cuda")
    g, f = _forward(nf, w, dev)
    rms = w.mode == W.RMSNORM
    H = w.hidden

    def outputs():
        return (torch.full_like(g["dy"], float("nan")),
                torch.full((H,), float("nan"), device=dev),
                None if rms else torch.full((H,), float("nan"), device=dev))

    dx_ref, dg_ref, db_ref = outputs()
    nf.ln_bwd(g["dy"], f["sum"], g["gamma"], f["mean"], f["rstd"], dx_ref, dg_ref, db_ref,
              mode=w.mode)
    torch.cuda.synchronize()
    scale = dx_row_scale(as_f64(g["dy"]), as_f64(g["gamma"]), as_f64(f["rstd"]), False)
    for _ in range(2):
        dx, dg, db = outputs()
        nf.ln_bwd_noalloc(g["dy"], f["sum"], g["gamma"], f["mean"], f["rstd"], dx, dg, db,
                          mode=w.mode)
        torch.cuda.synchronize()
        assert nf.ln_device_error() == 0
        check_elementwise(as_f64(dx), as_f64(dx_ref), w.dtype, "dx", scale_rows=scale)
        check_rel_l2(as_f64(dg), as_f64(dg_ref), 1e-4, "dgamma")
        if not rms:
            check_rel_l2(as_f64(db), as_f64(db_ref), 1e-4, "dbeta")


def test_noalloc_backward_reports_scratch_limit(cuda_lib):
    # LayerNorm at hidden 16384 with one row per CTA needs
    # 304 CTAs x 2 x 16384 x 4 bytes of partials, past the 16 MiB array.
    nf = cuda_lib
    lib = nf.load_library()
    rows, H = 400, 16384
    need = nf.ln_bwd_workspace_bytes(rows, H, torch.bfloat16, "layernorm")
    limit = 16 << 20
    assert need > limit
    dev = "cuda"
    t = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt, device=dev)
    dy, xs, gm, dx = t(rows, H), t(rows, H), t(H), t(rows, H)
    mean, rstd = t(rows, dt=torch.float32), t(rows, dt=torch.float32)
    dg, db = t(H, dt=torch.float32), t(H, dt=torch.float32)
    st = lib.ln_bwd_noalloc(dy.data_ptr(), xs.data_ptr(), gm.data_ptr(), mean.data_ptr(),
                            rstd.data_ptr(), dx.data_ptr(), dg.data_ptr(), db.data_ptr(),
                            None, rows, H, 1, 0, 0)
    assert st == 8, nf.ln_status_string(st)
    assert "SCRATCH_LIMIT" in nf.ln_status_string(st)
