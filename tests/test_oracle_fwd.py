"""Pins for the oracle's forward (bias + residual add, LayerNorm/RMSNorm, amax).

Independent anchors: torch's own fp64 ``layer_norm`` / ``rms_norm`` routines,
hand-derived worked examples in ``tests/golden``, closed forms for H = 1,
H = 2 and constant rows, and the invariants of the normalized row.
"""

import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import LAYERNORM, RMSNORM, norm_fwd, round_to_format

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _arr(v):
    return None if v is None else np.asarray(v, dtype=np.float64)


@pytest.mark.parametrize("name", ["ln_fwd_h4.json", "rms_fwd_h4.json",
                                  "ln_fwd_bf16_stored_sum.json"])
def test_golden_forward(name):
    g = json.load(open(os.path.join(GOLDEN, name)))
    out = norm_fwd(_arr(g["x"]), _arr(g["bias"]), _arr(g["residual"]), _arr(g["gamma"]),
                   _arr(g["beta"]), g["eps"], g["mode"], g["zero_centered_gamma"], g["fmt"])
    e = g["expect"]
    np.testing.assert_array_equal(out["sum"], _arr(e["sum"]))
    np.testing.assert_array_equal(out["rstd"], _arr(e["rstd"]))
    if "mean" in e:
        np.testing.assert_array_equal(out["mean"], _arr(e["mean"]))
    np.testing.assert_array_equal(out["y"], _arr(e["y"]))
    assert out["amax"] == e["amax"]


def _rand_case(rng, R, H, with_bias=True, with_res=True):
    x = rng.standard_normal((R, H)) * 1.5 + 0.3
    b = rng.standard_normal(H) * 0.2 if with_bias else None
    r = rng.standard_normal((R, H)) if with_res else None
    g = 1 + 0.3 * rng.standard_normal(H)
    be = 0.3 * rng.standard_normal(H)
    return x, b, r, g, be


@pytest.mark.parametrize("zc", [False, True])
@pytest.mark.parametrize("H", [1, 2, 7, 64, 384])
def test_layernorm_matches_torch_fp64(H, zc):
    rng = np.random.default_rng(10 + H)
    x, b, r, g, be = _rand_case(rng, 9, H)
    eps = 1e-5
    out = norm_fwd(x, b, r, g, be, eps, LAYERNORM, zc, "f64")
    s = torch.from_numpy((x + b[None, :]) + r)
    w = torch.from_numpy(1 + g if zc else g)
    want = F.layer_norm(s, (H,), w, torch.from_numpy(be), eps).numpy()
    np.testing.assert_allclose(out["y"], want, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(out["sum"], s.numpy())


@pytest.mark.parametrize("H", [1, 3, 64, 8192])
def test_rmsnorm_matches_torch_fp64(H):
    rng = np.random.default_rng(20 + H)
    x, b, r, g, _ = _rand_case(rng, 5, H, with_bias=False)
    eps = 1e-6
    out = norm_fwd(x, None, r, g, None, eps, RMSNORM, False, "f64")
    s = torch.from_numpy(x + r)
    want = F.rms_norm(s, (H,), torch.from_numpy(g), eps).numpy()
    np.testing.assert_allclose(out["y"], want, rtol=1e-12, atol=1e-12)
    assert out["mean"] is None


def test_zero_centered_gamma_equals_shifted_weight():
    rng = np.random.default_rng(30)
    x, b, r, g, be = _rand_case(rng, 6, 32)
    a = norm_fwd(x, b, r, g, be, 1e-5, LAYERNORM, True, "f64")
    c = norm_fwd(x, b, r, 1 + g, be, 1e-5, LAYERNORM, False, "f64")
    np.testing.assert_array_equal(a["y"], c["y"])


def test_normalized_row_invariants():
    # mean(xhat) = 0 and var(xhat) = var/(var + eps) for LayerNorm;
    # mean(xhat^2) = ms/(ms + eps) for RMSNorm.
    rng = np.random.default_rng(31)
    x, b, r, g, be = _rand_case(rng, 16, 384)
    eps = 1e-3
    ln = norm_fwd(x, b, r, g, be, eps, LAYERNORM, False, "f64")
    s = ln["sum"]
    var = s.var(axis=1)
    np.testing.assert_allclose(ln["xhat"].mean(axis=1), 0.0, atol=1e-13)
    np.testing.assert_allclose(ln["xhat"].var(axis=1), var / (var + eps), rtol=1e-12)
    rms = norm_fwd(x, b, r, g, None, eps, RMSNORM, False, "f64")
    ms = (s ** 2).mean(axis=1)
    np.testing.assert_allclose((rms["xhat"] ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-12)


def test_special_cases_h1_constant_row_h2():
    eps = 1e-5
    # H = 1: xhat = 0, y = beta, rstd = 1/sqrt(eps)
    out = norm_fwd(np.array([[3.0], [-7.0]]), None, None, np.array([2.0]), np.array([0.25]),
                   eps, LAYERNORM, False, "f64")
    np.testing.assert_array_equal(out["y"], [[0.25], [0.25]])
    np.testing.assert_allclose(out["rstd_exact"], [eps ** -0.5] * 2, rtol=1e-15)
    # constant row: variance 0, y = beta
    out = norm_fwd(np.full((1, 5), 1.75), None, None, np.arange(5.0), np.linspace(-1, 1, 5),
                   eps, LAYERNORM, False, "f64")
    np.testing.assert_array_equal(out["y"][0], np.linspace(-1, 1, 5))
    # H = 2 closed form: xhat = -+ (d/2) / sqrt(d^2/4 + eps), d = s1 - s0
    s0, s1 = 0.5, 2.0
    d = s1 - s0
    out = norm_fwd(np.array([[s0, s1]]), None, None, np.ones(2), np.zeros(2),
                   eps, LAYERNORM, False, "f64")
    v = (d / 2) / np.sqrt(d * d / 4 + eps)
    np.testing.assert_allclose(out["y"][0], [-v, v], rtol=1e-15)


def test_add_order_and_rounded_sum():
    # (x + bias) + residual, rounded once to the I/O format.
    rng = np.random.default_rng(32)
    x = round_to_format(rng.standard_normal((4, 16)), "bf16")
    b = round_to_format(rng.standard_normal(16) * 0.1, "bf16")
    r = round_to_format(rng.standard_normal((4, 16)), "bf16")
    out = norm_fwd(x, b, r, np.ones(16), np.zeros(16), 1e-5, LAYERNORM, False, "bf16")
    bits = torch.from_numpy((x + b[None, :]) + r).to(torch.float32).to(torch.bfloat16)
    np.testing.assert_array_equal(out["sum"], bits.to(torch.float64).numpy())


def test_amax_is_max_of_block_maxima():
    # The split of the full amax into per-block partial maxima plus a final
    # max (NVIDIA/Fuser issue 1660) gives the same value for any block split.
    rng = np.random.default_rng(33)
    x, b, r, g, be = _rand_case(rng, 40, 24)
    out = norm_fwd(x, b, r, g, be, 1e-5, LAYERNORM, False, "bf16")
    for block in (1, 3, 7, 40):
        parts = [np.abs(out["y"][i:i + block]).max() for i in range(0, 40, block)]
        assert max(parts) == out["amax"]
    assert out["amax"] == np.abs(out["y"]).max()
    assert norm_fwd(np.zeros((0, 4)), None, None, np.ones(4), None, 1e-5,
                    RMSNORM, False, "f32")["amax"] == 0.0


def test_statistics_rounded_to_fp32():
    rng = np.random.default_rng(34)
    x, b, r, g, be = _rand_case(rng, 8, 48)
    out = norm_fwd(x, b, r, g, be, 1e-5, LAYERNORM, False, "f32")
    np.testing.assert_array_equal(out["mean"], out["mean_exact"].astype(np.float32))
    np.testing.assert_array_equal(out["rstd"], out["rstd_exact"].astype(np.float32))
