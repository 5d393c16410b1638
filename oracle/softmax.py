"""Plain fp64 CPU oracle for the row softmax.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The product path
never touches it, and this module imports nothing from the product package.

What it computes (iree-org/iree issue 9139, the softmax IR after elementwise
fusion and the single-dispatch form that follows it): for every row of an
[R, H] matrix, over its H columns,

1. ``m = max_j x_j``, starting from -inf;
2. ``e_j = exp(x_j - m)``;
3. ``s = sum_j e_j``, starting from 0;
4. ``y_j = e_j / s``.

The issue fuses these four generic ops into one dispatch; the result is the
same four steps, which is what this module writes out. Inputs are decoded to
float64, every step runs in float64 with IEEE semantics (a row whose entries
are all -inf gives NaN, as ``-inf - (-inf)`` does), and only ``y`` is rounded
to the I/O format at the end.
"""

from __future__ import annotations

import numpy as np

from .norm import round_to_format


def softmax_fwd(x, fmt: str = "f64") -> dict:
    """Row softmax of a 2-D array.

    Returns ``y`` (rounded to ``fmt``: ``"f64"``, ``"f32"``, ``"bf16"`` or
    ``"f16"``), ``y_exact`` (float64), and the per-row ``max`` and ``sum``
    of step 1 and step 3.
    """
    x = np.asarray(x, dtype=np.float64)
    if x.ndim != 2:
        raise ValueError("softmax_fwd expects a 2-D [rows, hidden] array")
    rows, hidden = x.shape
    m = np.full(rows, -np.inf)
    if hidden:
        m = np.maximum(m, x.max(axis=1))
    with np.errstate(invalid="ignore"):
        e = np.exp(x - m[:, None])
    s = e.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        y = e / s[:, None]
    return {"y": round_to_format(y, fmt), "y_exact": y, "max": m, "sum": s}
