"""Pins for the oracle's backward (dx over hidden, dgamma/dbeta over rows).

Independent anchors: central finite differences of L = sum(dy * y) through
the oracle's forward, torch autograd in fp64, hand-derived worked examples,
closed-form row identities, the reordered-reduction identity of NVIDIA/Fuser
issue 1660, and split invariance of the outer reductions.
"""

import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import LAYERNORM, RMSNORM, norm_bwd, norm_fwd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _arr(v):
    return None if v is None else np.asarray(v, dtype=np.float64)


@pytest.mark.parametrize("name", ["ln_bwd_h4.json", "rms_bwd_h4.json"])
def test_golden_backward(name):
    g = json.load(open(os.path.join(GOLDEN, name)))
    out = norm_bwd(_arr(g["dy"]), _arr(g["x_sum"]), _arr(g["gamma"]), _arr(g["mean"]),
                   _arr(g["rstd"]), g["mode"], g["zero_centered_gamma"], g["fmt"])
    e = g["expect"]
    np.testing.assert_array_equal(out["dx"], _arr(e["dx"]))
    np.testing.assert_array_equal(out["dgamma"], _arr(e["dgamma"]))
    if e["dbeta"] is None:
        assert out["dbeta"] is None
    else:
        np.testing.assert_array_equal(out["dbeta"], _arr(e["dbeta"]))


def _case(seed, R=4, H=8):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((R, H)) + 0.5, bias=0.3 * rng.standard_normal(H),
                residual=rng.standard_normal((R, H)), gamma=1 + 0.4 * rng.standard_normal(H),
                beta=0.4 * rng.standard_normal(H), dy=rng.standard_normal((R, H)))


def _loss(c, mode, zc, eps):
    out = norm_fwd(c["x"], c["bias"], c["residual"], c["gamma"],
                   c["beta"] if mode == LAYERNORM else None, eps, mode, zc, "f64")
    return float((c["dy"] * out["y_exact"]).sum())


@pytest.mark.parametrize("zc", [False, True])
@pytest.mark.parametrize("mode", [LAYERNORM, RMSNORM])
def test_central_finite_differences(mode, zc):
    eps, h = 1e-5, 1e-6
    c = _case(40 + (mode == RMSNORM) + 2 * zc)
    fwd = norm_fwd(c["x"], c["bias"], c["residual"], c["gamma"],
                   c["beta"] if mode == LAYERNORM else None, eps, mode, zc, "f64")
    bwd = norm_bwd(c["dy"], fwd["sum"], c["gamma"], fwd["mean_exact"], fwd["rstd_exact"],
                   mode, zc, "f64")
    grads = {"x": bwd["dx_exact"], "residual": bwd["dx_exact"],
             "bias": bwd["dbias"], "gamma": bwd["dgamma"]}
    if mode == LAYERNORM:
        grads["beta"] = bwd["dbeta"]
    for name, want in grads.items():
        fd = np.zeros_like(c[name])
        for idx in np.ndindex(c[name].shape):
            cp = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in c.items()}
            cm = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in c.items()}
            cp[name][idx] += h
            cm[name][idx] -= h
            fd[idx] = (_loss(cp, mode, zc, eps) - _loss(cm, mode, zc, eps)) / (2 * h)
        scale = max(1.0, np.abs(want).max())
        np.testing.assert_allclose(fd, want, rtol=0, atol=1e-7 * scale, err_msg=name)


@pytest.mark.parametrize("zc", [False, True])
@pytest.mark.parametrize("mode", [LAYERNORM, RMSNORM])
def test_matches_torch_autograd_fp64(mode, zc):
    eps = 1e-6
    c = _case(50, R=12, H=96)
    fwd = norm_fwd(c["x"], c["bias"], c["residual"], c["gamma"],
                   c["beta"] if mode == LAYERNORM else None, eps, mode, zc, "f64")
    bwd = norm_bwd(c["dy"], fwd["sum"], c["gamma"], fwd["mean_exact"], fwd["rstd_exact"],
                   mode, zc, "f64")
    t = {k: torch.from_numpy(v).requires_grad_(True) for k, v in c.items() if k != "dy"}
    s = (t["x"] + t["bias"]) + t["residual"]
    w = 1 + t["gamma"] if zc else t["gamma"]
    if mode == LAYERNORM:
        y = F.layer_norm(s, (96,), w, t["beta"], eps)
    else:
        y = F.rms_norm(s, (96,), w, eps)
    (y * torch.from_numpy(c["dy"])).sum().backward()
    np.testing.assert_allclose(bwd["dx_exact"], t["x"].grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(bwd["dgamma"], t["gamma"].grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(bwd["dbias"], t["bias"].grad.numpy(), rtol=1e-10, atol=1e-12)
    if mode == LAYERNORM:
        np.testing.assert_allclose(bwd["dbeta"], t["beta"].grad.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", [LAYERNORM, RMSNORM])
def test_row_identities(mode):
    # LayerNorm: sum_j dx_j = 0. Both: sum_j dx_j xhat_j = rstd * eps/(v + eps) * sum_j g_j xhat_j,
    # v = variance (LayerNorm) or mean square (RMSNorm); with eps = 0 it vanishes.
    rng = np.random.default_rng(60)
    R, H = 16, 384
    xs, dy = rng.standard_normal((R, H)) * 2 + 1, rng.standard_normal((R, H))
    gamma = 1 + 0.1 * rng.standard_normal(H)
    for eps in (0.0, 0.5):
        if mode == LAYERNORM:
            mean, v = xs.mean(axis=1), xs.var(axis=1)
        else:
            mean, v = None, (xs ** 2).mean(axis=1)
        rstd = 1 / np.sqrt(v + eps)
        out = norm_bwd(dy, xs, gamma, mean, rstd, mode, False, "f64")
        dx, xhat = out["dx_exact"], out["xhat"]
        if mode == LAYERNORM:
            np.testing.assert_allclose(dx.sum(axis=1), 0.0, atol=1e-11)
        lhs = (dx * xhat).sum(axis=1)
        rhs = rstd * eps / (v + eps) * ((dy * gamma) * xhat).sum(axis=1)
        np.testing.assert_allclose(lhs, rhs, atol=1e-11)


def test_reordered_reduction_identity():
    # NVIDIA/Fuser issue 1660 toy: for x[8,4,1] and b[8,1,4], sum(x,1)*sum(b,1)
    # equals sum(x*b,1) because each operand is constant along the other's
    # reduced axis.
    rng = np.random.default_rng(70)
    x, b = rng.standard_normal((8, 4, 1)), rng.standard_normal((8, 1, 4))
    np.testing.assert_allclose(x.sum(axis=1) * b.sum(axis=1), (x * b).sum(axis=1), rtol=1e-13)
    # Applied to the dx reduction: mean and rstd are per-row broadcasts, so
    # mean_j(g * xhat) = rstd * (mean_j(g * x_sum) - mean * mean_j(g)).
    # Feed dx through that reordered c2 and compare with the oracle's dx.
    R, H = 8, 64
    xs, dy = rng.standard_normal((R, H)) + 3, rng.standard_normal((R, H))
    gamma = 1 + 0.1 * rng.standard_normal(H)
    mean, rstd = xs.mean(axis=1), 1 / np.sqrt(xs.var(axis=1) + 1e-5)
    out = norm_bwd(dy, xs, gamma, mean, rstd, LAYERNORM, False, "f64")
    g = dy * gamma
    c1 = g.mean(axis=1)
    c2_reordered = rstd * ((g * xs).mean(axis=1) - mean * c1)
    xhat = (xs - mean[:, None]) * rstd[:, None]
    dx_re = rstd[:, None] * (g - c1[:, None] - xhat * c2_reordered[:, None])
    np.testing.assert_allclose(out["dx_exact"], dx_re, rtol=1e-9, atol=1e-12)


def test_outer_reductions_split_invariance_and_column_sums():
    rng = np.random.default_rng(80)
    R, H = 37, 24
    xs, dy = rng.standard_normal((R, H)), rng.standard_normal((R, H))
    gamma = 1 + 0.1 * rng.standard_normal(H)
    mean, rstd = xs.mean(axis=1), 1 / np.sqrt(xs.var(axis=1) + 1e-5)
    full = norm_bwd(dy, xs, gamma, mean, rstd, LAYERNORM, False, "f64")
    # dbeta is the plain column sum of dy, by a scalar loop.
    for j in range(H):
        acc = 0.0
        for i in range(R):
            acc += dy[i, j]
        assert abs(full["dbeta"][j] - acc) <= 1e-12
    # any partition of the rows into blocks gives the same totals
    for block in (1, 5, 16):
        dg = np.zeros(H)
        db = np.zeros(H)
        for i in range(0, R, block):
            part = norm_bwd(dy[i:i + block], xs[i:i + block], gamma, mean[i:i + block],
                            rstd[i:i + block], LAYERNORM, False, "f64")
            dg += part["dgamma"]
            db += part["dbeta"]
        np.testing.assert_allclose(dg, full["dgamma"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(db, full["dbeta"], rtol=1e-12, atol=1e-12)


def test_h1_gives_zero_dx():
    out = norm_bwd(np.array([[2.0], [-1.0]]), np.array([[5.0], [1.0]]), np.array([3.0]),
                   np.array([5.0, 1.0]), np.array([300.0, 300.0]), LAYERNORM, False, "f64")
    np.testing.assert_array_equal(out["dx"], 0.0)
