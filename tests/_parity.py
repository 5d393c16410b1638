"""Helpers for the GPU parity tests: run the CUDA library through its C ABI
binding, run the oracle on the same inputs, and compare with the stated
tolerances.

Tolerances (per output):
* fp32 I/O: sum, y and dx max abs error <= 2e-5; rstd relative error <= 1e-5;
  mean error <= 1e-5 * mean_j |s_j| (the row's scale: a relative error of a
  mean that cancels to ~0 is not meaningful); dgamma/dbeta relative L2 error
  <= 1e-4.
* bf16/fp16 I/O: every element within 2 ulp of the oracle's value rounded to
  the dtype and >= 99.9 % within 1 ulp, the ulp taken at
  max(|ref|, 2^-8 * max_row |ref|) so that elements that cancel to ~0 are
  measured on the row's scale; the fp32 outputs (mean, rstd, dgamma, dbeta)
  use the fp32 rules.
* amax: bit-exact against max |y| over the kernel's own stored y.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import LAYERNORM, RMSNORM, norm_bwd, norm_fwd, round_to_format
from workloads import TORCH_DTYPES, as_f64

GUARD_BYTES = 4096
GUARD_BYTE = 0xA5
_P = {"f32": (24, -126), "bf16": (8, -126), "f16": (11, -14)}


class Guarded:
    """An output tensor with 4 KiB guard bands before and after it.

    The guards hold a byte pattern the kernels must not touch; the tensor
    itself starts as NaN (float) so any element the kernel fails to write
    shows up in the comparison.
    """

    def __init__(self, shape, dtype, device="cuda", fill=float("nan")):
        es = torch.empty(0, dtype=dtype).element_size()
        n = int(np.prod(shape)) if len(shape) else 1
        g = GUARD_BYTES // es
        self.g, self.n = g, n
        self.buf = torch.empty(n + 2 * g, dtype=dtype, device=device)
        self.buf.view(torch.uint8).fill_(GUARD_BYTE)
        self.t = self.buf[g:g + n].view(*shape)
        if n:
            self.t.fill_(fill)

    def guards_intact(self) -> bool:
        b = self.buf.view(torch.uint8)
        gb = self.g * self.buf.element_size()
        head, tail = b[:gb], b[b.numel() - gb:]
        return bool((head == GUARD_BYTE).all() and (tail == GUARD_BYTE).all())


def fmt_of(w) -> str:
    return w.dtype


def gpu_fwd(lib, w, inp, *, store_sum=True, stats=True, amax=None, stream=None,
            x_override=None):
    """Run ln_fwd on the workload's inputs; returns CPU tensors + guard status."""
    dev = "cuda"
    dt = TORCH_DTYPES[w.dtype]
    R, H = w.rows, w.hidden
    rms = w.mode == RMSNORM
    x = (x_override if x_override is not None else inp["x"]).to(dev)
    res = inp["residual"].to(dev) if inp["residual"] is not None else None
    bias = inp["bias"].to(dev) if inp["bias"] is not None else None
    gamma = inp["gamma"].to(dev)
    beta = inp["beta"].to(dev) if inp["beta"] is not None else None
    outs = {"y": Guarded((R, H), dt)}
    if store_sum:
        outs["sum"] = Guarded((R, H), dt)
    if stats:
        outs["rstd"] = Guarded((R,), torch.float32)
        if not rms:
            outs["mean"] = Guarded((R,), torch.float32)
    do_amax = w.amax if amax is None else amax
    if do_amax:
        outs["amax"] = Guarded((1,), torch.float32)
    g = {k: v.t for k, v in outs.items()}
    lib.ln_fwd(x, bias, res, gamma, beta, w.eps, w.mode, w.zero_centered_gamma,
               g.get("sum"), g["y"], g.get("mean"), g.get("rstd"), g.get("amax"), stream)
    torch.cuda.synchronize()
    assert lib.ln_device_error() == 0, "a kernel reported a failed wait"
    result = {k: v.t.cpu() for k, v in outs.items()}
    result["guards_ok"] = all(v.guards_intact() for v in outs.values())
    return result


def gpu_bwd(lib, w, dy, x_sum, gamma, mean, rstd, *, need_dbeta=True, need_dbias=False,
            grad_dtype=torch.float32, workspace=None, stream=None):
    """Run ln_bwd (ln_bwd_ex with dbias or a low-precision grad_dtype); inputs
    are CPU or CUDA tensors. Returns CPU tensors."""
    dev = "cuda"
    dt = TORCH_DTYPES[w.dtype]
    R, H = w.rows, w.hidden
    rms = w.mode == RMSNORM
    dy, x_sum, gamma = dy.to(dev), x_sum.to(dev), gamma.to(dev)
    mean = mean.to(dev) if (mean is not None and not rms) else None
    rstd = rstd.to(dev)
    outs = {"dx": Guarded((R, H), dt), "dgamma": Guarded((H,), grad_dtype)}
    if need_dbeta and not rms:
        outs["dbeta"] = Guarded((H,), grad_dtype)
    if need_dbias:
        outs["dbias"] = Guarded((H,), grad_dtype)
    g = {k: v.t for k, v in outs.items()}
    if need_dbias or grad_dtype != torch.float32:
        lib.ln_bwd_ex(dy, x_sum, gamma, mean, rstd, g["dx"], g["dgamma"], g.get("dbeta"),
                      g["dbias"], stream, mode=w.mode, zero_centered_gamma=w.zero_centered_gamma,
                      workspace=workspace)
    else:
        lib.ln_bwd(dy, x_sum, gamma, mean, rstd, g["dx"], g["dgamma"], g.get("dbeta"), stream,
                   mode=w.mode, zero_centered_gamma=w.zero_centered_gamma, workspace=workspace)
    torch.cuda.synchronize()
    assert lib.ln_device_error() == 0, "a kernel reported a failed wait"
    result = {k: v.t.cpu() for k, v in outs.items()}
    result["guards_ok"] = all(v.guards_intact() for v in outs.values())
    return result


def rows_f64(t, rows=None):
    """Rows of a CPU tensor (all, a slice or an index array) as float64 numpy."""
    if t is None:
        return None
    if rows is None:
        return as_f64(t)
    if isinstance(rows, slice):
        return as_f64(t[rows])
    return as_f64(t[torch.as_tensor(np.asarray(rows), dtype=torch.long)])


def oracle_fwd(w, inp, rows=None, x_override=None):
    x = x_override if x_override is not None else inp["x"]
    return norm_fwd(rows_f64(x, rows), as_f64(inp["bias"]), rows_f64(inp["residual"], rows),
                    as_f64(inp["gamma"]), as_f64(inp["beta"]), w.eps, w.mode,
                    w.zero_centered_gamma, w.dtype)


def oracle_bwd_rows(w, dy, x_sum, gamma, mean, rstd, rows):
    return norm_bwd(rows_f64(dy, rows), rows_f64(x_sum, rows), as_f64(gamma),
                    rows_f64(mean, rows), rows_f64(rstd, rows), w.mode,
                    w.zero_centered_gamma, w.dtype)


def oracle_bwd_reductions(w, dy, x_sum, gamma, mean, rstd, chunk=32768):
    """dgamma, dbeta over every row; the oracle runs on row blocks and the
    block results are added (the outer reductions are sums over rows)."""
    R = dy.shape[0]
    dg = np.zeros(w.hidden)
    db = None if w.mode == RMSNORM else np.zeros(w.hidden)
    g64 = as_f64(gamma)
    for i in range(0, R, chunk):
        sl = slice(i, min(R, i + chunk))
        m = None if mean is None else as_f64(mean[sl])
        o = norm_bwd(as_f64(dy[sl]), as_f64(x_sum[sl]), g64, m, as_f64(rstd[sl]), w.mode,
                     w.zero_centered_gamma, w.dtype)
        dg += o["dgamma"]
        if db is not None:
            db += o["dbeta"]
    return dg, db


def oracle_stats_full(w, x, chunk=32768):
    """fp32 mean/rstd of the oracle's forward over every row (no add)."""
    R = x.shape[0]
    mean = np.zeros(R, dtype=np.float32) if w.mode == LAYERNORM else None
    rstd = np.zeros(R, dtype=np.float32)
    ones = np.ones(w.hidden)
    for i in range(0, R, chunk):
        sl = slice(i, min(R, i + chunk))
        o = norm_fwd(as_f64(x[sl]), None, None, ones, None, w.eps, w.mode, False, w.dtype)
        rstd[sl] = o["rstd"]
        if mean is not None:
            mean[sl] = o["mean"]
    return (None if mean is None else torch.from_numpy(mean)), torch.from_numpy(rstd)


def ulp(mag: np.ndarray, fmt: str) -> np.ndarray:
    """Spacing of ``fmt`` at magnitude ``mag`` (subnormal spacing below the normals)."""
    p, emin = _P[fmt]
    mag = np.asarray(mag, dtype=np.float64)
    _, E = np.frexp(mag)
    e = np.where(mag > 0, np.maximum(E - 1, emin), emin)
    return np.ldexp(1.0, e - (p - 1))


def dx_row_scale(dy_rows, gamma, rstd_rows, zero_centered_gamma: bool) -> np.ndarray:
    """Per-row size of the terms dx is the difference of: rstd * max_j |dy_j w_j|.

    dx = rstd * (g - c1 - xhat * c2) cancels to far below its terms when the
    row is short and eps is small against the variance (H = 1 RMSNorm gives
    dx = rstd * g * eps / (s^2 + eps)); fp32 arithmetic then carries an error
    of ~1e-7 of the terms, which is what the ulp floor is measured against.
    """
    w = np.asarray(gamma, dtype=np.float64)
    w = 1.0 + w if zero_centered_gamma else w
    g = np.abs(np.asarray(dy_rows, dtype=np.float64) * w[None, :])
    return np.asarray(rstd_rows, dtype=np.float64) * g.max(axis=1)


def check_elementwise(got, ref_exact, fmt: str, what: str, row_scale=True, scale_rows=None,
                      max_floored=None):
    """Apply the dtype's element tolerance; returns a short report dict.

    ``scale_rows`` (optional, per row) replaces max_row |ref| as the row
    scale of the ulp floor. The report also gives the same counts without
    the floor (ulp taken at |ref| alone): ``worst_ulp_raw``, ``within1_raw``
    and ``floored``, the number of elements more than 2 ulp off by that plain
    rule, i.e. the elements the row-scale floor decided. With
    ``max_floored`` set, their fraction must not pass it, so an error that
    hides behind the floor fails loudly."""
    got = np.asarray(got, dtype=np.float64)
    ref_exact = np.asarray(ref_exact, dtype=np.float64)
    assert got.shape == ref_exact.shape, (what, got.shape, ref_exact.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    if got.size == 0:
        return {"what": what, "n": 0}
    if fmt == "f32":
        err = np.abs(got - ref_exact).max()
        assert err <= 2e-5, f"{what}: max abs error {err:.3e} > 2e-5"
        return {"what": what, "max_abs": float(err)}
    ref_r = round_to_format(ref_exact, fmt)
    diff = np.abs(got - ref_r)
    mag_raw = np.abs(ref_exact)
    d_raw = diff / ulp(mag_raw, fmt)
    mag = mag_raw
    if row_scale and ref_exact.ndim == 2:
        rs = np.max(mag_raw, axis=1) if scale_rows is None else np.maximum(
            np.max(mag_raw, axis=1), np.asarray(scale_rows, dtype=np.float64))
        mag = np.maximum(mag_raw, np.ldexp(rs, -8)[:, None])
    d = diff / ulp(mag, fmt)
    worst = float(d.max())
    within1 = float((d <= 1.0).mean())
    floored = int((d_raw > 2.0).sum())
    report = {"what": what, "n": int(d.size), "worst_ulp": worst, "within1": within1,
              "worst_ulp_raw": float(d_raw.max()), "within1_raw": float((d_raw <= 1.0).mean()),
              "floored": floored, "floored_frac": floored / d.size}
    assert worst <= 2.0, f"{what}: worst {worst:.2f} ulp > 2"
    assert within1 >= 0.999, f"{what}: only {within1:.5f} within 1 ulp"
    if max_floored is not None:
        assert report["floored_frac"] <= max_floored, (
            f"{what}: {floored} of {d.size} elements pass only through the row-scale floor "
            f"(> {max_floored:g}): {report}")
    return report


def check_mean(got, mean_exact, sum_rows, what="mean"):
    """Mean error within 1e-5 of the row's scale mean_j |s_j|; returns how
    many rows that rule decided (more than 1e-5 off relative to |mean|
    itself, which means nothing for a mean that cancels to ~0)."""
    got = np.asarray(got, dtype=np.float64)
    scale = np.abs(np.asarray(sum_rows, dtype=np.float64)).mean(axis=1)
    err = np.abs(got - mean_exact)
    ok = err <= 1e-5 * np.maximum(scale, np.finfo(np.float32).tiny)
    assert ok.all(), f"{what}: worst {float((err / np.maximum(scale, 1e-30)).max()):.3e} of row scale"
    decided = int((err > 1e-5 * np.abs(mean_exact)).sum())
    return {"what": what, "n": int(err.size), "row_scale_decided": decided,
            "row_scale_decided_frac": decided / max(err.size, 1)}


def check_rel(got, ref, tol, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), np.finfo(np.float32).tiny)
    assert rel.max() <= tol, f"{what}: max rel error {rel.max():.3e} > {tol}"


def check_rel_l2(got, ref, tol, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.linalg.norm(got - ref)
    den = np.linalg.norm(ref)
    rel = num / den if den > 0 else num
    assert rel <= tol, f"{what}: relative L2 error {rel:.3e} > {tol}"
    return rel


def amax_bits_of(y: torch.Tensor) -> int:
    """fp32 bit pattern of max |y| over a stored tensor, computed on the host."""
    if y.numel() == 0:
        return 0
    a = np.abs(as_f64(y)).astype(np.float32)
    return int(a.view(np.uint32).max())


def amax_bits_got(t: torch.Tensor) -> int:
    return int(t.cpu().numpy().astype(np.float32).view(np.uint32)[0])
