"""Pins for the oracle's row softmax.

Independent anchors: a hand-derived worked example (tests/golden), SciPy's
and torch's own fp64 softmax, scalar ``math.exp`` brute force on tiny rows,
the closed forms for constant and masked rows, and the invariants (rows sum
to one, a per-row shift changes nothing). A dropped max subtraction, a sum
over the wrong axis or a division by the wrong quantity fails at least one.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import round_to_format
from oracle import softmax_fwd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _arr(rows):
    # float() also parses the strings "-inf" and "nan" the fixture uses
    return np.array([[float(v) for v in r] for r in rows], dtype=np.float64)


def test_golden_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "softmax_h4.json")))
    out = softmax_fwd(_arr(g["x"]), g["fmt"])
    want = _arr(g["expect"]["y"])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(out["y"]), nan)
    np.testing.assert_allclose(out["y"][~nan], want[~nan], rtol=0, atol=g["tol"])


def test_matches_scipy_softmax():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(90)
    x = rng.standard_normal((37, 129)) * np.array([0.1, 1, 5, 30])[rng.integers(0, 4, 37)][:, None]
    np.testing.assert_allclose(softmax_fwd(x)["y"], special.softmax(x, axis=1), rtol=1e-13,
                               atol=1e-300)


def test_matches_torch_softmax_fp64_non_square():
    rng = np.random.default_rng(91)
    x = rng.standard_normal((5, 300)) * 4 + 2
    want = torch.softmax(torch.from_numpy(x), dim=1).numpy()
    np.testing.assert_allclose(softmax_fwd(x)["y"], want, rtol=1e-13, atol=1e-300)


def test_brute_force_scalar_loops():
    rng = np.random.default_rng(92)
    x = rng.standard_normal((3, 7)) * 3
    got = softmax_fwd(x)
    for i in range(3):
        m = max(x[i])
        e = [math.exp(v - m) for v in x[i]]
        s = math.fsum(e)
        assert got["max"][i] == m
        assert abs(got["sum"][i] - s) <= 1e-14 * s
        for j in range(7):
            assert abs(got["y"][i, j] - e[j] / s) <= 1e-15


def test_invariants_sum_to_one_and_shift():
    rng = np.random.default_rng(93)
    x = rng.standard_normal((64, 513)) * 3
    y = softmax_fwd(x)["y"]
    np.testing.assert_allclose(y.sum(axis=1), 1.0, atol=1e-13)
    shift = rng.standard_normal(64)[:, None] * 50
    np.testing.assert_allclose(softmax_fwd(x + shift)["y"], y, rtol=1e-11, atol=1e-300)
    # ratios: y_i / y_j = exp(x_i - x_j)
    np.testing.assert_allclose(y[:, 0] / y[:, 1], np.exp(x[:, 0] - x[:, 1]), rtol=1e-12)


def test_closed_forms():
    np.testing.assert_array_equal(softmax_fwd(np.full((2, 8), 3.5))["y"], 0.125)
    np.testing.assert_array_equal(softmax_fwd(np.array([[7.0]]))["y"], [[1.0]])
    out = softmax_fwd(np.zeros((3, 0)))
    assert out["y"].shape == (3, 0)


def test_rounding_to_io_formats_is_one_rounding_of_the_exact_value():
    rng = np.random.default_rng(94)
    x = rng.standard_normal((8, 200)) * 2
    out = softmax_fwd(x, "f16")
    # numpy's float64 -> float16 cast is a single correct rounding
    np.testing.assert_array_equal(out["y"], out["y_exact"].astype(np.float16).astype(np.float64))
    out = softmax_fwd(x, "f32")
    np.testing.assert_array_equal(out["y"], out["y_exact"].astype(np.float32).astype(np.float64))
    np.testing.assert_array_equal(softmax_fwd(x, "bf16")["y"],
                                  round_to_format(out["y_exact"], "bf16"))
