"""Plain fp64 CPU oracle for the fused normalization block.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The product path
(the CUDA library and its Python binding) never touches it, and this module
imports nothing from the product package.

What it computes, and where the definition comes from:

* Forward (NVIDIA/Fuser issue 1660, the "layernorm + amax" snippet):
  ``out1 = (x + bias) + residual``; ``w = ln_weight`` or ``1 + ln_weight``
  when ``zero_centered_gamma``; ``out2 = layer_norm(out1, w, ln_bias, eps)``;
  ``amax = max |out2|``. The mean -> variance -> normalize split of the
  LayerNorm forward, with the variance depending on the mean and the
  normalize step reading the input again, is the one iree-org/iree issue 9139
  discusses (its opening comment and the comparison with softmax further
  down). RMSNorm is named on pytorch/pytorch PR 165370 but never defined
  there; the textbook definition is used.
* Backward (pytorch/pytorch PR 165370, the two kinds of reduction in an
  RMS/Layer norm backward): dx reduces over the hidden dimension, dw/db
  reduce over the B x T rows.

Readings where the pages are silent (each is listed with its reason in the
design notes):

* A: the statistics are taken from the sum *as stored* in the I/O dtype,
  because the snippet materialises ``out1`` before ``layer_norm`` reads it.
* B: LayerNorm variance is the biased one (divide by H), ``eps`` inside the
  square root; RMSNorm is ``y = s * rstd * w`` with
  ``rstd = 1 / sqrt(mean(s^2) + eps)``, no mean and no beta.
* C: ``1 + ln_weight`` is formed in full precision, not rounded to the I/O
  dtype first.
* D: the add order is ``(x + bias) + residual``; absent operands count as 0.
* E: the backward takes mean and rstd as inputs (fp32 values), exactly as
  the kernel does.

Everything is vectorised numpy in float64 and follows the definitions term by
term: no blocking, no fusion, no reordering of the sums beyond numpy's own
row reductions.
"""

from __future__ import annotations

import numpy as np

LAYERNORM = "layernorm"
RMSNORM = "rmsnorm"

# (precision bits incl. the implicit one, minimum normal exponent, maximum exponent)
_FORMATS = {
    "f32": (24, -126, 127),
    "bf16": (8, -126, 127),
    "f16": (11, -14, 15),
}


def round_to_format(v, fmt: str) -> np.ndarray:
    """Round float64 values to the nearest value of ``fmt``, ties to even.

    ``fmt`` is one of ``"f64"`` (identity), ``"f32"``, ``"bf16"``, ``"f16"``.
    The result is returned as float64 holding exactly representable values.
    Subnormals of the target format are produced on its fixed subnormal grid;
    values past the largest finite number round to +-inf as IEEE 754
    round-to-nearest-even does.
    """
    v = np.asarray(v, dtype=np.float64)
    if fmt == "f64":
        return v.copy()
    p, emin, emax = _FORMATS[fmt]
    out = v.copy()
    finite = np.isfinite(v) & (v != 0.0)
    vf = v[finite]
    # v = m * 2**E with 0.5 <= |m| < 1, so floor(log2 |v|) = E - 1 exactly.
    _, E = np.frexp(vf)
    e = np.maximum(E - 1, emin)
    quantum_exp = e - (p - 1)
    q = np.ldexp(vf, -quantum_exp)  # exact: scaling by a power of two
    r = np.ldexp(np.rint(q), quantum_exp)  # np.rint rounds half to even
    max_finite = np.ldexp(2.0 - 2.0 ** (1 - p), emax)
    r = np.where(np.abs(r) > max_finite, np.copysign(np.inf, vf), r)
    # keep the sign of values that round to zero
    r = np.where(r == 0.0, np.copysign(0.0, vf), r)
    out[finite] = r
    return out


E4M3_MAX = 448.0


def round_to_e4m3_satfinite(v) -> np.ndarray:
    """Round float64 values to FP8 E4M3 (1 sign, 4 exponent bits with bias 7,
    3 mantissa bits; no infinities), nearest even, saturating finite values
    beyond the largest finite magnitude (448) to +-448; NaN stays NaN.

    E4M3 has normals from 2**-6 and subnormals spaced 2**-9; 1.875 * 2**8
    would be the next value after 448 but that pattern is NaN, so a value that
    rounds past 448 saturates to it."""
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    finite = np.isfinite(v) & (v != 0.0)
    vf = v[finite]
    _, E = np.frexp(vf)
    e = np.maximum(E - 1, -6)
    quantum_exp = e - 3
    r = np.ldexp(np.rint(np.ldexp(vf, -quantum_exp)), quantum_exp)
    r = np.clip(r, -E4M3_MAX, E4M3_MAX)
    r = np.where(r == 0.0, np.copysign(0.0, vf), r)
    out[finite] = r
    out[np.isinf(v)] = np.copysign(E4M3_MAX, v[np.isinf(v)])
    return out


def quantize_fp8_e4m3(y_stored, scale: float) -> np.ndarray:
    """The FP8 output of the forward: the stored y times the per-tensor
    scale, multiplied in fp32 (the precision the kernel takes the decision
    in), then rounded to E4M3 with saturation. The scale is the caller's
    (delayed scaling: typically 448 / the amax of an earlier step)."""
    prod = round_to_format(np.asarray(y_stored, dtype=np.float64) *
                           float(np.float32(scale)), "f32")
    return round_to_e4m3_satfinite(prod)


def _weight(gamma: np.ndarray, zero_centered_gamma: bool) -> np.ndarray:
    """w = ln_weight, or 1 + ln_weight for zero-centered gamma (Fuser 1660)."""
    gamma = np.asarray(gamma, dtype=np.float64)
    return 1.0 + gamma if zero_centered_gamma else gamma


def norm_fwd(x, bias, residual, gamma, beta, eps: float, mode: str,
             zero_centered_gamma: bool, fmt: str) -> dict:
    """Forward of the fused block on a [rows, H] float64 array.

    Inputs hold values already representable in ``fmt`` (decoded to float64).
    ``bias``, ``residual`` and ``beta`` may be None. Returns a dict with

    * ``sum``: rnd(s) with s = (x + bias) + residual, the stored add result;
    * ``y``: rnd(y_exact); ``y_exact``: the unrounded normalized output;
    * ``mean`` (LayerNorm only, else None) and ``rstd``, rounded to fp32,
      plus ``mean_exact`` / ``rstd_exact`` in float64;
    * ``amax``: max |y| over the rounded outputs (0 for an empty input).
    """
    x = np.asarray(x, dtype=np.float64)
    if x.ndim != 2:
        raise ValueError("x must be [rows, H]")
    rows, H = x.shape
    # F1: out1 = (x + bias) + residual, stored in the I/O dtype.
    s = x.copy()
    if bias is not None:
        s = s + np.asarray(bias, dtype=np.float64)[None, :]
    if residual is not None:
        s = s + np.asarray(residual, dtype=np.float64)
    out_sum = round_to_format(s, fmt)
    shat = out_sum  # reading A: statistics of the stored sum
    # F2: statistics over the hidden dimension.
    if mode == LAYERNORM:
        mean = shat.mean(axis=1)
        var = ((shat - mean[:, None]) ** 2).mean(axis=1)
        rstd = 1.0 / np.sqrt(var + eps)
    elif mode == RMSNORM:
        mean = None
        ms = (shat ** 2).mean(axis=1)
        rstd = 1.0 / np.sqrt(ms + eps)
    else:
        raise ValueError(f"unknown mode {mode!r}")
    # F3: normalize and affine.
    w = _weight(gamma, zero_centered_gamma)
    if mode == LAYERNORM:
        xhat = (shat - mean[:, None]) * rstd[:, None]
        y_exact = xhat * w[None, :]
        if beta is not None:
            y_exact = y_exact + np.asarray(beta, dtype=np.float64)[None, :]
    else:
        xhat = shat * rstd[:, None]
        y_exact = xhat * w[None, :]
    y = round_to_format(y_exact, fmt)
    # F4: amax of |y| over the whole tensor (Fuser 1660, the FP8 amax step).
    amax = float(np.max(np.abs(y))) if y.size else 0.0
    return {
        "sum": out_sum,
        "y": y,
        "y_exact": y_exact,
        "xhat": xhat,
        "mean": None if mean is None else round_to_format(mean, "f32"),
        "rstd": round_to_format(rstd, "f32"),
        "mean_exact": mean,
        "rstd_exact": rstd,
        "amax": amax,
    }


def norm_bwd(dy, x_sum, gamma, mean, rstd, mode: str,
             zero_centered_gamma: bool, fmt: str) -> dict:
    """Backward of the fused block given the forward's saved statistics.

    ``x_sum`` is the stored sum (the normalization input), ``mean`` and
    ``rstd`` the per-row statistics the forward produced (``mean`` is None for
    RMSNorm). Returns

    * ``dx``: rnd(dx_exact), the gradient with respect to the normalization
      input (and so, through the identity add, to x and to residual);
      ``dx_exact`` unrounded;
    * ``dgamma``: sum over rows of dy * xhat (float64);
    * ``dbeta``: sum over rows of dy (float64; None for RMSNorm);
    * ``dbias``: sum over rows of dx_exact, the gradient of the bias through
      the forward's add (float64).

    With xhat = (x_sum - mean) * rstd (RMSNorm: x_sum * rstd), g = dy * w,
    c1 = mean_j g, c2 = mean_j g * xhat, the inner (per-row) reduction is
    dx = rstd * (g - c1 - xhat * c2), with c1 dropped for RMSNorm. The outer
    reductions over rows give dgamma and dbeta (PR 165370). d w / d gamma = 1
    for both gamma conventions, so dgamma has the same expression.
    """
    dy = np.asarray(dy, dtype=np.float64)
    x_sum = np.asarray(x_sum, dtype=np.float64)
    rstd = np.asarray(rstd, dtype=np.float64)
    w = _weight(gamma, zero_centered_gamma)
    if mode == LAYERNORM:
        mean = np.asarray(mean, dtype=np.float64)
        xhat = (x_sum - mean[:, None]) * rstd[:, None]
    elif mode == RMSNORM:
        xhat = x_sum * rstd[:, None]
    else:
        raise ValueError(f"unknown mode {mode!r}")
    g = dy * w[None, :]
    # B1: inner reduction over the hidden dimension.
    c2 = (g * xhat).mean(axis=1)
    if mode == LAYERNORM:
        c1 = g.mean(axis=1)
        dx_exact = rstd[:, None] * (g - c1[:, None] - xhat * c2[:, None])
    else:
        dx_exact = rstd[:, None] * (g - xhat * c2[:, None])
    dx = round_to_format(dx_exact, fmt)
    # B2/B3: outer reductions over the rows.
    dgamma = (dy * xhat).sum(axis=0)
    dbeta = dy.sum(axis=0) if mode == LAYERNORM else None
    # The forward adds bias to every row, so its gradient is the column sum
    # of the gradient of the normalization input (Fuser 1660's add feeding
    # the norm whose backward PR 165370 fuses).
    dbias = dx_exact.sum(axis=0)
    return {"dx": dx, "dx_exact": dx_exact, "dgamma": dgamma, "dbeta": dbeta,
            "dbias": dbias, "xhat": xhat}
