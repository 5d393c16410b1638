"""GPU parity of ln_fwd_from_partials (the normalize step fed by per-tile
partial statistics, NVIDIA/cutlass discussion 874, example 37's
gemm_with_layernorm) against the oracle's ``norm_fwd_from_partials``.

The partials stand in for what a GEMM epilogue would emit: the oracle's
``row_tile_partials`` of the stored row, summed in fp64 and rounded to fp32.
Both sides take those fp32 values as given. Checked: y element by element
(the dtype's ulp rule: LayerNorm's row-scale floor share recorded and
bounded, RMSNorm's y held to the plain rule), rstd (relative 1e-5), mean
(1e-5 of the row's scale), amax bit-exact against the kernel's own y, guard
bands untouched. Shapes cover the lane-group
kernel, the CTA-per-row kernel and the scalar kernel, ragged row tails and
ragged last tiles, both partial forms, both modes and zero-centered gamma.
"""

import numpy as np
import pytest
import torch

import workloads as W
from _parity import Guarded, amax_bits_got, amax_bits_of, check_elementwise, check_mean, check_rel
from oracle import norm_fwd_from_partials, row_tile_partials
from workloads import Workload, as_f64, make_inputs

pytestmark = pytest.mark.gpu


def _case(name, dtype, rows, hidden, mode, zc=False):
    return Workload(name=name, dtype=dtype, rows=rows, hidden=hidden, mode=mode, eps=1e-5,
                    x_std=1.0, gamma_std=0.05, beta_std=0.05 if mode == W.LAYERNORM else None,
                    zero_centered_gamma=zc, backward=False)


CASES = [
    (_case("p_bf16_4133x384", "bf16", 4133, 384, W.LAYERNORM), 128),       # lane groups, T = 3
    (_case("p_bf16_4133x384_rms", "bf16", 4133, 384, W.RMSNORM), 96),
    (_case("p_bf16_1000x768_zc", "bf16", 1000, 768, W.LAYERNORM, zc=True), 100),  # ragged tile
    (_case("p_f16_777x1280", "f16", 777, 1280, W.LAYERNORM), 96),
    (_case("p_f32_513x384", "f32", 513, 384, W.LAYERNORM), 64),
    (_case("p_bf16_300x8192", "bf16", 300, 8192, W.LAYERNORM), 128),       # CTA per row, T = 64
    (_case("p_bf16_300x8192_rms", "bf16", 300, 8192, W.RMSNORM), 1000),
    (_case("p_bf16_211x2560", "bf16", 211, 2560, W.LAYERNORM), 128),       # 64-thread CTA, 5 vectors
    (_case("p_bf16_97x3000_rms", "bf16", 97, 3000, W.RMSNORM), 256),       # fitted CTA, idle slots
    (_case("p_bf16_257x1001", "bf16", 257, 1001, W.LAYERNORM), 128),       # scalar kernel
    (_case("p_f32_64x5", "f32", 64, 5, W.LAYERNORM), 2),
]


def run_partials(lib, w, tile, kind, inp, amax=True):
    dev = "cuda"
    dt = W.TORCH_DTYPES[w.dtype]
    R, H = w.rows, w.hidden
    x64 = as_f64(inp["x"])
    psum, psq = row_tile_partials(x64, tile, kind, fmt="f32")
    ps = torch.from_numpy(psum.astype(np.float32)).to(dev)
    pq = torch.from_numpy(psq.astype(np.float32)).to(dev)
    rms = w.mode == W.RMSNORM
    outs = {"y": Guarded((R, H), dt), "rstd": Guarded((R,), torch.float32)}
    if not rms:
        outs["mean"] = Guarded((R,), torch.float32)
    if amax:
        outs["amax"] = Guarded((1,), torch.float32)
    g = {k: v.t for k, v in outs.items()}
    beta = inp["beta"].to(dev) if inp["beta"] is not None else None
    lib.ln_fwd_from_partials(inp["x"].to(dev), ps, pq, tile, kind, inp["gamma"].to(dev), beta,
                             w.eps, w.mode, w.zero_centered_gamma, g["y"], g.get("mean"),
                             g["rstd"], g.get("amax"))
    torch.cuda.synchronize()
    got = {k: v.t.cpu() for k, v in outs.items()}
    got["guards_ok"] = all(v.guards_intact() for v in outs.values())
    ref = norm_fwd_from_partials(x64, psum, psq, tile, kind, as_f64(inp["gamma"]),
                                 as_f64(inp["beta"]), w.eps, w.mode, w.zero_centered_gamma,
                                 w.dtype)
    return got, ref


@pytest.mark.parametrize("w,tile", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
@pytest.mark.parametrize("kind", ["sum_sq", "sum_m2"])
def test_from_partials_matches_oracle(cuda_lib, w, tile, kind, record_property):
    inp = make_inputs(w, seed=31)
    got, ref = run_partials(cuda_lib, w, tile, kind, inp)
    assert got["guards_ok"]
    rep = check_elementwise(as_f64(got["y"]), ref["y_exact"], w.dtype, "y",
                            row_scale=w.mode == W.LAYERNORM, max_floored=1e-3)
    for k in ("floored", "floored_frac"):
        if k in rep:
            record_property(f"y_{k}", rep[k])
    check_rel(as_f64(got["rstd"]), ref["rstd_exact"], 1e-5, "rstd")
    if w.mode == W.LAYERNORM:
        check_mean(as_f64(got["mean"]), ref["mean_exact"], as_f64(inp["x"]))
    assert amax_bits_got(got["amax"]) == amax_bits_of(got["y"])


def test_from_partials_matches_the_fused_forward_statistics(cuda_lib):
    """Partials of the stored sum that ln_fwd writes give the statistics
    ln_fwd computed itself, within fp32 rounding (the same row, two routes)."""
    w = W.BENCH_LN_BF16_576000x384.with_(rows=2049, backward=False)
    inp = make_inputs(w, seed=5)
    dev = "cuda"
    g = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    f = cuda_lib.fused_norm_fwd(g["x"], g["gamma"], g["beta"], bias=g["bias"],
                                residual=g["residual"], eps=w.eps, store_sum=True)
    s64 = as_f64(f["sum"].cpu())
    for kind in ("sum_sq", "sum_m2"):
        psum, psq = row_tile_partials(s64, 128, kind, fmt="f32")
        p = cuda_lib.fused_norm_fwd_from_partials(
            f["sum"], torch.from_numpy(psum.astype(np.float32)).to(dev),
            torch.from_numpy(psq.astype(np.float32)).to(dev), 128, g["gamma"], g["beta"],
            kind=kind, eps=w.eps)
        torch.cuda.synchronize()
        check_rel(as_f64(p["rstd"].cpu()), as_f64(f["rstd"].cpu()), 2e-6, f"rstd {kind}")
        scale = np.abs(s64).mean(axis=1)
        assert (np.abs(as_f64(p["mean"].cpu()) - as_f64(f["mean"].cpu())) <= 1e-6 * scale).all()


def test_from_partials_zero_rows_and_one_tile(cuda_lib):
    w = _case("p_bf16_0x384", "bf16", 0, 384, W.LAYERNORM)
    inp = make_inputs(w, seed=1)
    got, _ = run_partials(cuda_lib, w, 128, "sum_sq", inp)
    assert got["guards_ok"] and float(got["amax"][0]) == 0.0
    w = _case("p_bf16_40x384", "bf16", 40, 384, W.LAYERNORM)
    inp = make_inputs(w, seed=2)
    for tile in (384, 5000):    # one tile either way
        got, ref = run_partials(cuda_lib, w, tile, "sum_m2", inp)
        check_elementwise(as_f64(got["y"]), ref["y_exact"], w.dtype, "y")


@pytest.mark.parametrize("hidden,tile", [(384, 128), (8192, 128), (1001, 100)])
def test_from_partials_m2_with_a_large_mean(cuda_lib, hidden, tile):
    """(Σ, M2) partials of rows s = 64 + N(0, 1), the variance ~1e-4 of the
    mean square: the parallel-variance combination takes no difference of
    large sums, so every output stays within the parity tolerances (the
    (Σ, Σ²) form's Q/H - mean² in fp32 would lose most of the variance's
    digits on such rows)."""
    w = _case(f"p_bf16_200x{hidden}_offset", "bf16", 200, hidden, W.LAYERNORM)
    inp = make_inputs(w, seed=41)
    inp = dict(inp, x=(inp["x"].double() + 64.0).to(torch.bfloat16))
    got, ref = run_partials(cuda_lib, w, tile, "sum_m2", inp)
    assert got["guards_ok"]
    check_elementwise(as_f64(got["y"]), ref["y_exact"], w.dtype, "y", max_floored=1e-3)
    check_rel(as_f64(got["rstd"]), ref["rstd_exact"], 1e-5, "rstd")
    check_mean(as_f64(got["mean"]), ref["mean_exact"], as_f64(inp["x"]))
    assert amax_bits_got(got["amax"]) == amax_bits_of(got["y"])
