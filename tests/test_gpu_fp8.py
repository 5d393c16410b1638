"""GPU parity of the FP8 (E4M3) copy of y written by ln_fwd_ex.

The decision the kernel takes, E4M3(fp32(y_stored * scale)) of its own
stored y, is checked bit for bit against the oracle's ``quantize_fp8_e4m3``
applied to that stored y (both take the product in fp32, the precision the
kernel decides in), with torch's float32 -> float8_e4m3fn cast (clamped to
+-448, the saturating cast) as a second opinion. Against the oracle's own y
(which the kernel's y may differ from by the ulp the bf16/fp16 rules allow,
moving a code by one step): >= 99.9 % of codes equal and every code within
one E4M3 step.
"""

import numpy as np
import pytest
import torch

import workloads as W
from _parity import Guarded, oracle_fwd
from oracle import E4M3_MAX, quantize_fp8_e4m3
from workloads import Workload, as_f64, make_inputs

pytestmark = pytest.mark.gpu


def e4m3_step(mag):
    mag = np.asarray(mag, dtype=np.float64)
    _, E = np.frexp(mag)
    e = np.where(mag > 0, np.maximum(E - 1, -6), -6)
    return np.ldexp(1.0, e - 3)


def run_fp8(lib, w, inp, scale_value, with_y=True):
    dev = "cuda"
    dt = W.TORCH_DTYPES[w.dtype]
    R, H = w.rows, w.hidden
    g = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    y = Guarded((R, H), dt) if with_y else None
    q = Guarded((R, H), torch.uint8, fill=0)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    scale = torch.tensor([scale_value], dtype=torch.float32, device=dev)
    rstd = torch.empty(R, dtype=torch.float32, device=dev)
    lib.ln_fwd_ex(g["x"], g["bias"], g["residual"], g["gamma"], g["beta"], w.eps, w.mode,
                  w.zero_centered_gamma, None, y.t if y is not None else None, None, rstd, amax,
                  q.t, scale)
    torch.cuda.synchronize()
    assert lib.ln_device_error() == 0
    assert q.guards_intact() and (y is None or y.guards_intact())
    return (y.t.cpu() if y is not None else None), q.t.cpu(), float(amax.cpu()[0])


def decode(codes: torch.Tensor) -> np.ndarray:
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


CASES = [
    W.FWD_AMAX_BF16_32768x768,
    W.UNET_F16[640].with_(rows=4099),
    W.LN_F32_4096x384,
    W.RMS_BF16_16384x8192.with_(rows=1500, outlier_frac=0.0),     # CTA-per-row kernel
    Workload(name="fp8_scalar_bf16_777x1001", dtype="bf16", rows=777, hidden=1001,
             mode=W.LAYERNORM, eps=1e-5, residual_std=1.0, bias_std=0.1, gamma_std=0.1,
             beta_std=0.1),                                          # scalar kernel
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("scale", [64.0, 300.0])   # 300 saturates the tail of |y|
def test_fp8_output(cuda_lib, w, scale):
    inp = make_inputs(w, seed=21)
    y, q, amax = run_fp8(cuda_lib, w, inp, scale)
    got = decode(q)
    # bit-exact: the oracle's E4M3 of the kernel's own stored y (value and
    # sign, which together fix the code of a non-NaN E4M3 number) ...
    want_own = quantize_fp8_e4m3(as_f64(y), scale)
    np.testing.assert_array_equal(got, want_own)
    np.testing.assert_array_equal(np.signbit(got), np.signbit(want_own))
    # ... and torch's saturating cast of the same product agrees
    prod = y.to(torch.float32) * torch.tensor(scale, dtype=torch.float32)
    want_t = prod.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, want_t)
    # against the oracle's y
    ref = oracle_fwd(w, inp)
    want = quantize_fp8_e4m3(ref["y"], scale)
    steps = np.abs(got - want) / e4m3_step(np.maximum(np.abs(want), 2.0 ** -6))
    assert steps.max() <= 1.0, steps.max()
    assert (got == want).mean() >= 0.999
    assert (np.abs(got) == E4M3_MAX).any() == (scale * np.abs(ref["y"]).max() >= E4M3_MAX)
    assert amax == float(np.abs(as_f64(y)).max())


def test_fp8_only_output_matches(cuda_lib):
    w = W.FWD_AMAX_BF16_32768x768.with_(rows=5001)
    inp = make_inputs(w, seed=22)
    y, q1, a1 = run_fp8(cuda_lib, w, inp, 100.0, with_y=True)
    none, q2, a2 = run_fp8(cuda_lib, w, inp, 100.0, with_y=False)
    assert none is None
    assert torch.equal(q1, q2) and a1 == a2
