"""Plain fp64 oracle of the normalize step fed by per-tile partial statistics.

TEST INFRASTRUCTURE ONLY (the same rule as ``oracle.norm``): only the tests,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may import it.

NVIDIA/cutlass discussion 874 (the reply that points at example 37,
``gemm_with_layernorm.h``): the GEMM that produces the row also computes, in
its epilogue, partial sums of the row's values over the column tile each
threadblock owns, so the LayerNorm that follows reads statistics instead of
taking a reduction pass over the row. The producer (the GEMM) is outside this
project; this module is the consumer's definition, the statistics combined
from the partials plainly, in the pages' order: the tile sums first, then
mean, then variance, then normalize.

Two partial forms (readings where the page names none: the plain epilogue
sums, and the form that keeps the variance well conditioned):

* ``"sum_sq"``: per row r and column tile t, ``psum[r, t] = sum_j s_j`` and
  ``psq[r, t] = sum_j s_j**2`` over the tile's columns. LayerNorm:
  ``mean = S / H``, ``var = Q / H - mean**2`` with ``S``, ``Q`` the sums over
  the tiles (floored at 0: rounding of the partials can push it below).
  RMSNorm: ``ms = Q / H``.
* ``"sum_m2"``: ``psum`` as above and ``psq[r, t] = sum_j (s_j - m_t)**2``
  with ``m_t = psum[r, t] / n_t`` the tile's own mean over its ``n_t``
  columns. The tiles combine by the parallel-variance identity (Chan, Golub
  and LeVeque, 1979): ``M2 = sum_t psq_t + sum_t n_t (m_t - mean)**2``,
  ``var = M2 / H``. RMSNorm: ``ms = sum_t (psq_t + n_t m_t**2) / H``.

Column tiles are ``tile_cols`` wide from column 0; the last one holds the
``H - (T - 1) * tile_cols`` columns left, ``T = ceil(H / tile_cols)``.
"""

from __future__ import annotations

import numpy as np

from .norm import LAYERNORM, RMSNORM, _weight, round_to_format

SUM_SQ = "sum_sq"
SUM_M2 = "sum_m2"


def tile_widths(H: int, tile_cols: int) -> np.ndarray:
    """n_t of every column tile of a row of H columns."""
    if tile_cols < 1:
        raise ValueError("tile_cols must be >= 1")
    T = -(-H // tile_cols)
    n = np.full(T, tile_cols, dtype=np.int64)
    n[-1] = H - (T - 1) * tile_cols
    return n


def row_tile_partials(s_stored, tile_cols: int, kind: str, fmt: str = "f32"):
    """The partials a producer would emit for the stored rows ``s_stored``
    ([rows, H] float64): fp64 sums over each column tile, rounded to ``fmt``
    ("f32", the epilogue's accumulator type, or "f64" to keep them exact).
    Returns (psum, psq), each [rows, T]."""
    s = np.asarray(s_stored, dtype=np.float64)
    rows, H = s.shape
    n = tile_widths(H, tile_cols)
    T = n.size
    psum = np.zeros((rows, T))
    psq = np.zeros((rows, T))
    for t in range(T):
        blk = s[:, t * tile_cols:t * tile_cols + n[t]]
        psum[:, t] = blk.sum(axis=1)
        if kind == SUM_SQ:
            psq[:, t] = (blk ** 2).sum(axis=1)
        elif kind == SUM_M2:
            m_t = psum[:, t] / n[t]
            psq[:, t] = ((blk - m_t[:, None]) ** 2).sum(axis=1)
        else:
            raise ValueError(f"unknown partial kind {kind!r}")
    return round_to_format(psum, fmt), round_to_format(psq, fmt)


def combine_partials(psum, psq, tile_cols: int, H: int, kind: str, mode: str):
    """Row statistics from the partials, in float64: (mean or None, var or
    mean square) per row, as the module docstring states."""
    psum = np.asarray(psum, dtype=np.float64)
    psq = np.asarray(psq, dtype=np.float64)
    n = tile_widths(H, tile_cols).astype(np.float64)
    if psum.shape[1] != n.size or psq.shape != psum.shape:
        raise ValueError("partials must be [rows, ceil(H / tile_cols)]")
    S = psum.sum(axis=1)
    mean = S / H
    if kind == SUM_SQ:
        Q = psq.sum(axis=1)
        if mode == RMSNORM:
            return None, Q / H
        return mean, np.maximum(Q / H - mean ** 2, 0.0)
    if kind == SUM_M2:
        m_t = psum / n[None, :]
        if mode == RMSNORM:
            return None, (psq + n[None, :] * m_t ** 2).sum(axis=1) / H
        M2 = psq.sum(axis=1) + (n[None, :] * (m_t - mean[:, None]) ** 2).sum(axis=1)
        return mean, M2 / H
    raise ValueError(f"unknown partial kind {kind!r}")


def norm_fwd_from_partials(x_stored, psum, psq, tile_cols: int, kind: str, gamma, beta,
                           eps: float, mode: str, zero_centered_gamma: bool,
                           fmt: str) -> dict:
    """Normalize the stored rows with statistics combined from the partials.

    ``x_stored`` [rows, H] holds the row as the producer stored it (values of
    ``fmt``); ``psum``/``psq`` [rows, T] the partials (their values taken as
    given). Returns ``y`` (rounded to fmt), ``y_exact``, ``mean``/``rstd``
    rounded to fp32, ``mean_exact``/``rstd_exact`` and ``amax`` of the
    rounded y, like ``norm_fwd``."""
    x = np.asarray(x_stored, dtype=np.float64)
    rows, H = x.shape
    mean, v = combine_partials(psum, psq, tile_cols, H, kind, mode)
    rstd = 1.0 / np.sqrt(v + eps)
    w = _weight(gamma, zero_centered_gamma)
    if mode == LAYERNORM:
        y_exact = (x - mean[:, None]) * rstd[:, None] * w[None, :]
        if beta is not None:
            y_exact = y_exact + np.asarray(beta, dtype=np.float64)[None, :]
    elif mode == RMSNORM:
        y_exact = x * rstd[:, None] * w[None, :]
    else:
        raise ValueError(f"unknown mode {mode!r}")
    y = round_to_format(y_exact, fmt)
    return {
        "y": y,
        "y_exact": y_exact,
        "mean": None if mean is None else round_to_format(mean, "f32"),
        "rstd": round_to_format(rstd, "f32"),
        "mean_exact": mean,
        "rstd_exact": rstd,
        "amax": float(np.max(np.abs(y))) if y.size else 0.0,
    }
