"""Plausible slips planted in the norm and softmax oracles fail their pins.

Each mutation edits one expression of oracle/norm.py (a copy of its source,
executed as a separate module; the oracle itself is untouched) and the pins
below run against the mutated copy. Every mutation must fail at least one
pin; the unmutated oracle must pass all of them. The pins do not reuse the
oracle's arithmetic: torch's fp64 layer_norm and autograd, the RMSNorm
formula written out, the stored sum formed here, a constant row's closed
form, and amax of the rounded output; for the rounding helpers, numpy's
fp16/fp32 casts, torch's bf16 and E4M3 casts and a constructed FP8 tie; for
the softmax, torch's fp64 softmax
on rows whose logits sit far above and below zero, and fully masked rows.
(The partials oracle has its own planted-slip test in test_oracle_partials.)
"""

import os
import types

import numpy as np
import pytest
import torch

import oracle.norm as R

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "oracle", "norm.py")).read()

# (name, text in oracle/norm.py, replacement)
MUTATIONS = [
    ("unbiased variance", "var = ((shat - mean[:, None]) ** 2).mean(axis=1)",
     "var = ((shat - mean[:, None]) ** 2).sum(axis=1) / (H - 1)"),
    ("eps outside the root", "rstd = 1.0 / np.sqrt(var + eps)",
     "rstd = 1.0 / (np.sqrt(var) + eps)"),
    ("RMSNorm centred", "ms = (shat ** 2).mean(axis=1)",
     "ms = ((shat - shat.mean(axis=1)[:, None]) ** 2).mean(axis=1)"),
    ("zero-centered gamma ignored", "return 1.0 + gamma if zero_centered_gamma else gamma",
     "return gamma"),
    ("beta dropped", "y_exact = y_exact + np.asarray(beta, dtype=np.float64)[None, :]",
     "y_exact = y_exact"),
    ("statistics of the unrounded sum", "shat = out_sum  # reading A", "shat = s  # reading A"),
    ("bias added twice", "s = s + np.asarray(bias, dtype=np.float64)[None, :]",
     "s = s + 2.0 * np.asarray(bias, dtype=np.float64)[None, :]"),
    ("amax of the unrounded y", "amax = float(np.max(np.abs(y))) if y.size else 0.0",
     "amax = float(np.max(np.abs(y_exact))) if y.size else 0.0"),
    ("c1 sign", "dx_exact = rstd[:, None] * (g - c1[:, None] - xhat * c2[:, None])",
     "dx_exact = rstd[:, None] * (g + c1[:, None] - xhat * c2[:, None])"),
    ("c2 term dropped", "dx_exact = rstd[:, None] * (g - c1[:, None] - xhat * c2[:, None])",
     "dx_exact = rstd[:, None] * (g - c1[:, None])"),
    ("RMSNorm keeps c1", "dx_exact = rstd[:, None] * (g - xhat * c2[:, None])",
     "dx_exact = rstd[:, None] * (g - g.mean(axis=1)[:, None] - xhat * c2[:, None])"),
    ("c2 without w", "c2 = (g * xhat).mean(axis=1)", "c2 = (dy * xhat).mean(axis=1)"),
    ("rstd outside the bracket", "dx_exact = rstd[:, None] * (g - c1[:, None] - xhat * c2[:, None])",
     "dx_exact = g - c1[:, None] - xhat * c2[:, None]"),
    ("dgamma from g", "dgamma = (dy * xhat).sum(axis=0)", "dgamma = (g * xhat).sum(axis=0)"),
    ("dbeta over the wrong axis", "dbeta = dy.sum(axis=0) if mode == LAYERNORM else None",
     "dbeta = dy.sum(axis=1) if mode == LAYERNORM else None"),
    ("xhat misparenthesised", "xhat = (x_sum - mean[:, None]) * rstd[:, None]",
     "xhat = x_sum * rstd[:, None] - mean[:, None]"),
    ("dbias of the rounded dx", "dbias = dx_exact.sum(axis=0)", "dbias = dx.sum(axis=0)"),
]


def mutated(old, new):
    assert SRC.count(old) == 1, old
    m = types.ModuleType("oracle_norm_mutant")
    exec(compile(SRC.replace(old, new), "oracle_norm_mutant", "exec"), m.__dict__)
    return m


def _inputs(seed, rows=6, H=16, fmt="bf16"):
    rng = np.random.default_rng(seed)
    rnd = lambda a: R.round_to_format(a, fmt)
    x = rnd(3.0 + rng.standard_normal((rows, H)))   # an offset, so the centring matters
    bias = rnd(0.3 * rng.standard_normal(H))
    res = rnd(rng.standard_normal((rows, H)))
    gamma = rnd(0.2 * rng.standard_normal(H))
    beta = rnd(0.2 * rng.standard_normal(H))
    dy = rnd(rng.standard_normal((rows, H)))
    return x, bias, res, gamma, beta, dy


def _stored_sum(x, bias, res, fmt="bf16"):
    return R.round_to_format((x + bias[None, :]) + res, fmt)


def _ref_forward(s, w, beta, eps, mode):
    """fp64 forward from the stored sum: torch layer_norm, or RMSNorm written out."""
    st = torch.tensor(s, dtype=torch.float64)
    wt = torch.tensor(w, dtype=torch.float64)
    if mode == R.LAYERNORM:
        return torch.nn.functional.layer_norm(st, (st.shape[1],), wt,
                                              torch.tensor(beta, dtype=torch.float64), eps)
    return st * torch.rsqrt((st * st).mean(dim=1, keepdim=True) + eps) * wt


def pin_forward(M):
    eps = 1e-3
    for mode in (R.LAYERNORM, R.RMSNORM):
        for zc in (False, True):
            x, bias, res, gamma, beta, _ = _inputs(1)
            out = M.norm_fwd(x, bias, res, gamma, beta if mode == R.LAYERNORM else None, eps,
                             mode, zc, "bf16")
            s = _stored_sum(x, bias, res)
            assert np.array_equal(out["sum"], s)
            w = 1.0 + gamma if zc else gamma
            ref = _ref_forward(s, w, beta, eps, mode).numpy()
            assert np.allclose(out["y_exact"], ref, rtol=1e-12, atol=1e-12)
            assert out["amax"] == float(np.max(np.abs(R.round_to_format(ref, "bf16"))))


def pin_constant_row(M):
    H = 16
    x = np.full((2, H), 1.5)
    gamma = np.linspace(0.5, 1.5, H)
    beta = np.linspace(-1.0, 1.0, H)
    out = M.norm_fwd(x, None, None, gamma, beta, 1e-5, R.LAYERNORM, False, "f32")
    assert np.array_equal(out["y_exact"], np.broadcast_to(beta, (2, H)))


def pin_backward(M):
    eps = 1e-3
    for mode in (R.LAYERNORM, R.RMSNORM):
        for zc in (False, True):
            x, bias, res, gamma, beta, dy = _inputs(2)
            s = _stored_sum(x, bias, res)
            # autograd through the forward from the stored sum; the statistics
            # the backward is given are the exact fp64 ones
            st = torch.tensor(s, dtype=torch.float64, requires_grad=True)
            gt = torch.tensor(gamma, dtype=torch.float64, requires_grad=True)
            bt = torch.tensor(beta, dtype=torch.float64, requires_grad=True)
            wt = 1.0 + gt if zc else gt
            if mode == R.LAYERNORM:
                y = torch.nn.functional.layer_norm(st, (st.shape[1],), wt, bt, eps)
            else:
                y = st * torch.rsqrt((st * st).mean(dim=1, keepdim=True) + eps) * wt
            (y * torch.tensor(dy, dtype=torch.float64)).sum().backward()
            sd = st.detach()
            if mode == R.LAYERNORM:
                mean = sd.mean(dim=1).numpy()
                rstd = torch.rsqrt(sd.var(dim=1, unbiased=False) + eps).numpy()
            else:
                mean = None
                rstd = torch.rsqrt((sd * sd).mean(dim=1) + eps).numpy()
            out = M.norm_bwd(dy, s, gamma, mean, rstd, mode, zc, "bf16")
            assert np.allclose(out["dx_exact"], st.grad.numpy(), rtol=1e-10, atol=1e-10)
            assert np.allclose(out["dgamma"], gt.grad.numpy(), rtol=1e-10, atol=1e-10)
            if mode == R.LAYERNORM:
                assert np.allclose(out["dbeta"], bt.grad.numpy(), rtol=1e-10, atol=1e-10)
            # the bias is added to every row, so its gradient is the column sum of dx
            assert np.allclose(out["dbias"], st.grad.numpy().sum(axis=0), rtol=1e-12,
                               atol=1e-12)


PINS = [pin_forward, pin_constant_row, pin_backward]


def _failures(M):
    failed = []
    for pin in PINS:
        try:
            pin(M)
        except Exception:   # an assertion, or a shape error the slip causes
            failed.append(pin.__name__)
    return failed


def test_the_oracle_passes_every_pin():
    assert _failures(R) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_each_planted_slip_fails_a_pin(name, old, new):
    assert _failures(mutated(old, new)), f"no pin caught: {name}"


# ---- the softmax oracle -------------------------------------------------------

import oracle.softmax as S   # noqa: E402

SMX_SRC = open(os.path.join(ROOT, "oracle", "softmax.py")).read().replace(
    "from .norm import round_to_format", "from oracle.norm import round_to_format")

SMX_MUTATIONS = [
    ("no max shift", "e = np.exp(x - m[:, None])", "e = np.exp(x)"),
    ("max from 0", "m = np.full(rows, -np.inf)", "m = np.zeros(rows)"),
    ("sum over the wrong axis", "s = e.sum(axis=1)", "s = e.sum(axis=0)"),
    ("divided by the max", "y = e / s[:, None]", "y = e / e.max(axis=1)[:, None]"),
]


def smx_mutated(old, new):
    assert SMX_SRC.count(old) == 1, old
    m = types.ModuleType("oracle_softmax_mutant")
    exec(compile(SMX_SRC.replace(old, new), "oracle_softmax_mutant", "exec"), m.__dict__)
    return m


def smx_pin_torch(M):
    rng = np.random.default_rng(3)
    x = 3.0 * rng.standard_normal((5, 12))
    x[1] += 800.0          # exp overflows without the max shift
    x[2] -= 800.0          # and underflows when the shift starts from 0
    x[3, ::3] = -np.inf    # masked entries
    ref = torch.softmax(torch.tensor(x, dtype=torch.float64), dim=1).numpy()
    got = M.softmax_fwd(x)["y_exact"]
    assert np.allclose(got, ref, rtol=1e-13, atol=0)
    assert (got[3, ::3] == 0).all()


def smx_pin_masked_row(M):
    x = np.zeros((2, 8))
    x[0, :] = -np.inf
    y = M.softmax_fwd(x)["y_exact"]
    assert np.isnan(y[0]).all() and np.allclose(y[1], 1.0 / 8)


def _smx_failures(M):
    failed = []
    for pin in (smx_pin_torch, smx_pin_masked_row):
        try:
            pin(M)
        except Exception:
            failed.append(pin.__name__)
    return failed


def test_the_softmax_oracle_passes_every_pin():
    assert _smx_failures(S) == []


@pytest.mark.parametrize("name,old,new", SMX_MUTATIONS, ids=[m[0] for m in SMX_MUTATIONS])
def test_each_planted_softmax_slip_fails_a_pin(name, old, new):
    assert _smx_failures(smx_mutated(old, new)), f"no pin caught: {name}"


# ---- the rounding helpers of the norm oracle ----------------------------------

ROUND_MUTATIONS = [
    ("ties away from zero", "r = np.ldexp(np.rint(q), quantum_exp)",
     "r = np.ldexp(np.sign(q) * np.floor(np.abs(q) + 0.5), quantum_exp)"),
    ("no subnormal grid", "e = np.maximum(E - 1, emin)", "e = E - 1"),
    ("one bit short", "quantum_exp = e - (p - 1)", "quantum_exp = e - p"),
    ("overflow kept finite",
     "r = np.where(np.abs(r) > max_finite, np.copysign(np.inf, vf), r)", "r = r"),
    ("E4M3 without saturation", "r = np.clip(r, -E4M3_MAX, E4M3_MAX)", "r = r"),
    ("E4M3 without subnormals", "e = np.maximum(E - 1, -6)", "e = E - 1"),
    ("FP8 product kept in fp64",
     'prod = round_to_format(np.asarray(y_stored, dtype=np.float64) *\n'
     '                           float(np.float32(scale)), "f32")',
     'prod = np.asarray(y_stored, dtype=np.float64) * float(np.float32(scale))'),
]


def _round_values():
    rng = np.random.default_rng(4)
    v = np.concatenate([
        rng.standard_normal(2000) * np.exp2(rng.integers(-30, 30, 2000)),
        [1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 1 + 2.0 ** -24, -(1 + 2.0 ** -24),   # ties
         2.0 ** -20, 3.1e-5, 2.0 ** -140, 7e-46,                               # subnormal ranges
         70000.0, 3.5e38, -1e39]])                                            # past the maxima
    return v


def rnd_pin_numpy_casts(M):
    v = _round_values()
    with np.errstate(over="ignore"):
        assert np.array_equal(M.round_to_format(v, "f16"), v.astype(np.float16).astype(np.float64))
        assert np.array_equal(M.round_to_format(v, "f32"), v.astype(np.float32).astype(np.float64))


def rnd_pin_bf16_torch(M):
    v32 = _round_values().astype(np.float32)
    v32 = v32[np.isfinite(v32)]
    ref = torch.tensor(v32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(M.round_to_format(v32.astype(np.float64), "bf16"), ref)


def rnd_pin_e4m3(M):
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.uniform(-448, 448, 3000), rng.uniform(-1, 1, 1000) * 2.0 ** -7,
                        [2.0 ** -9, 3 * 2.0 ** -10, 0.0]])
    ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).double().numpy()
    got = M.round_to_e4m3_satfinite(v.astype(np.float32).astype(np.float64))
    assert np.array_equal(got, ref)
    big = np.array([449.0, 480.0, 1e6, -1e6, np.inf, -np.inf])
    assert np.array_equal(M.round_to_e4m3_satfinite(big), np.sign(big) * 448.0)


def _fp32_tie_case():
    """A bf16 y and an fp32 scale whose exact product lies just above the
    E4M3 tie 1.0625 (between 1 and 1.125) while its fp32 rounding is the tie
    itself, which rounds to even (1.0): the fp32 product decides."""
    for k in range(1, 128):
        y0 = 1.0 + k / 128.0                      # bf16 values in (1, 2)
        sc = float(np.float32(1.0625 / y0))
        exact = y0 * sc
        if exact > 1.0625 and float(np.float32(exact)) == 1.0625:
            return y0, sc
    raise AssertionError("no tie case found")


def rnd_pin_fp8_product(M):
    rng = np.random.default_rng(6)
    y = M.round_to_format(rng.standard_normal(4000), "bf16")
    scale = 37.3
    prod = torch.tensor(y, dtype=torch.float32) * torch.tensor(scale, dtype=torch.float32)
    ref = prod.clamp(-448, 448).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(M.quantize_fp8_e4m3(y, scale), ref)
    y0, sc = _fp32_tie_case()
    assert M.quantize_fp8_e4m3(np.array([y0]), sc)[0] == 1.0


ROUND_PINS = [rnd_pin_numpy_casts, rnd_pin_bf16_torch, rnd_pin_e4m3, rnd_pin_fp8_product]


def _round_failures(M):
    failed = []
    for pin in ROUND_PINS:
        try:
            pin(M)
        except Exception:
            failed.append(pin.__name__)
    return failed


def test_the_rounding_helpers_pass_every_pin():
    assert _round_failures(R) == []


@pytest.mark.parametrize("name,old,new", ROUND_MUTATIONS, ids=[m[0] for m in ROUND_MUTATIONS])
def test_each_planted_rounding_slip_fails_a_pin(name, old, new):
    assert _round_failures(mutated(old, new)), f"no pin caught: {name}"
