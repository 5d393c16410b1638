"""Seeded synthetic inputs for the fused normalization block.

This module holds random draws and their conversion to the I/O dtype, and
nothing of the normalization arithmetic. Both the tests (for the oracle and
the CUDA library alike) and ``bench.py`` take their inputs from here.

Recipe (the same for every workload):

* one ``numpy.random.Generator(PCG64(seed))`` per workload;
* tensors are drawn in this order, each only if the workload has it:
  x, outlier positions, residual, bias, gamma, beta, dy;
* a draw ``std * N(0, 1)`` is made in float64, rounded to float32
  (round-to-nearest-even), then to bf16/fp16 (round-to-nearest-even) when the
  workload's dtype is one of those;
* gamma is ``1 + gamma_std * N(0, 1)``, except for zero-centered gamma where
  the stored tensor is ``gamma_std * N(0, 1)`` (the weight then is 1 + gamma);
* outliers: ``round(frac * rows * hidden)`` distinct flat positions drawn with
  ``Generator.choice(..., replace=False)``; x at those positions is scaled
  by ``outlier_scale`` before rounding.

Tensors are returned on the CPU, contiguous, in the workload's dtype.
"""

from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
LAYERNORM = "layernorm"
RMSNORM = "rmsnorm"


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "f32" | "bf16" | "f16"
    rows: int
    hidden: int
    mode: str             # "layernorm" | "rmsnorm"
    eps: float
    x_std: float = 1.0
    residual_std: float | None = None   # None: no residual operand
    bias_std: float | None = None       # None: no bias operand
    gamma_std: float = 0.0
    beta_std: float | None = None       # None: no beta (always None for RMSNorm)
    zero_centered_gamma: bool = False
    amax: bool = False
    backward: bool = True                # draw dy
    forward: bool = True
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    fp8_out: bool = False                # the step also writes an E4M3 copy of y
    dbias: bool = False                  # the step's backward also writes dbias

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# Shapes and distributions of the five configurations the block is checked
# and measured on. The 576000 x 384 shape is the (1152 * 500, 384) norm
# backward of pytorch/pytorch PR 165370; 384 and 768 are miniLM/BERT-class
# hidden sizes (iree-org/iree issue 9139); 320/640/1280 are the stable
# diffusion UNet widths behind NVIDIA/cutlass discussion 874.
LN_F32_4096x384 = Workload(
    name="ln_f32_4096x384", dtype="f32", rows=4096, hidden=384, mode=LAYERNORM,
    eps=1e-5, x_std=1.0, residual_std=1.0, bias_std=0.1, gamma_std=0.1,
    beta_std=0.1)

BWD_BF16_576000x384_LN = Workload(
    name="bwd_ln_bf16_576000x384", dtype="bf16", rows=576000, hidden=384,
    mode=LAYERNORM, eps=1e-6, x_std=1.0, gamma_std=0.02, beta_std=0.02,
    forward=False)
BWD_BF16_576000x384_RMS = BWD_BF16_576000x384_LN.with_(
    name="bwd_rms_bf16_576000x384", mode=RMSNORM, beta_std=None)

FWD_AMAX_BF16_32768x768 = Workload(
    name="fwd_amax_bf16_32768x768", dtype="bf16", rows=32768, hidden=768,
    mode=LAYERNORM, eps=1e-5, x_std=1.0, residual_std=1.0, bias_std=0.1,
    gamma_std=0.02, beta_std=0.02, zero_centered_gamma=True, amax=True,
    backward=False)

UNET_F16 = {
    h: Workload(name=f"unet_ln_f16_8192x{h}", dtype="f16", rows=8192, hidden=h,
                mode=LAYERNORM, eps=1e-5, x_std=2.0, residual_std=1.0,
                gamma_std=0.05, beta_std=0.05)
    for h in (320, 640, 1280)
}

RMS_BF16_16384x8192 = Workload(
    name="rms_bf16_16384x8192", dtype="bf16", rows=16384, hidden=8192,
    mode=RMSNORM, eps=1e-6, x_std=1.0, residual_std=0.5, gamma_std=0.02,
    outlier_frac=0.001, outlier_scale=100.0)

# The step bench.py times: the whole fused forward (bias + residual add,
# LayerNorm, amax) and the fused backward at the 576000 x 384 bf16 shape.
BENCH_LN_BF16_576000x384 = Workload(
    name="ln_fwd_bwd_bf16_576000x384", dtype="bf16", rows=576000, hidden=384,
    mode=LAYERNORM, eps=1e-6, x_std=1.0, residual_std=1.0, bias_std=0.1,
    gamma_std=0.02, beta_std=0.02, amax=True)
BENCH_RMS_BF16_16384x8192 = RMS_BF16_16384x8192.with_(
    name="rms_fwd_bwd_bf16_16384x8192", amax=True)
# The same step with the options of the next rows of the scope table: an
# FP8 (E4M3) copy of y scaled from a per-tensor scale, and dbias.
BENCH_LN_FP8_DBIAS_BF16_576000x384 = BENCH_LN_BF16_576000x384.with_(
    name="ln_fwd_bwd_fp8_dbias_bf16_576000x384", fp8_out=True, dbias=True)
# The normalize step fed by per-column-tile partial statistics, on the
# 576000 x 384 rows with 128-column tiles (three tiles per row).
PARTIALS_BF16_576000x384 = BENCH_LN_BF16_576000x384.with_(
    name="partials_bf16_576000x384", residual_std=None, bias_std=None, backward=False)
PARTIALS_TILE_COLS = 128

WORKLOADS = {w.name: w for w in (
    LN_F32_4096x384, BWD_BF16_576000x384_LN, BWD_BF16_576000x384_RMS,
    FWD_AMAX_BF16_32768x768, *UNET_F16.values(), RMS_BF16_16384x8192,
    BENCH_LN_BF16_576000x384, BENCH_RMS_BF16_16384x8192, BENCH_LN_FP8_DBIAS_BF16_576000x384,
    PARTIALS_BF16_576000x384)}


def to_dtype(a64: np.ndarray, dtype: str) -> torch.Tensor:
    """float64 -> float32 (RNE) -> bf16/fp16 (RNE), as a contiguous CPU tensor."""
    t = torch.from_numpy(np.ascontiguousarray(a64, dtype=np.float32))
    if dtype != "f32":
        t = t.to(TORCH_DTYPES[dtype])
    return t.contiguous()


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw the workload's tensors. Keys absent from the workload map to None."""
    rng = np.random.Generator(np.random.PCG64(seed))
    R, H = w.rows, w.hidden
    x = w.x_std * rng.standard_normal((R, H))
    if w.outlier_frac > 0.0 and R * H > 0:
        k = int(round(w.outlier_frac * R * H))
        pos = rng.choice(R * H, size=k, replace=False)
        x.reshape(-1)[pos] *= w.outlier_scale
    out = {"x": to_dtype(x, w.dtype)}
    del x
    out["residual"] = (to_dtype(w.residual_std * rng.standard_normal((R, H)), w.dtype)
                       if w.residual_std is not None else None)
    out["bias"] = (to_dtype(w.bias_std * rng.standard_normal(H), w.dtype)
                   if w.bias_std is not None else None)
    g = w.gamma_std * rng.standard_normal(H)
    out["gamma"] = to_dtype(g if w.zero_centered_gamma else 1.0 + g, w.dtype)
    out["beta"] = (to_dtype(w.beta_std * rng.standard_normal(H), w.dtype)
                   if (w.beta_std is not None and w.mode == LAYERNORM) else None)
    out["dy"] = (to_dtype(rng.standard_normal((R, H)), w.dtype)
                 if w.backward else None)
    return out


# ---- row softmax ------------------------------------------------------------
# The softmax IR of iree-org/iree issue 9139 is a 6 x 3 fp32 toy with an
# elided constant, so no shape or distribution comes from the pages. The
# softmax workloads reuse the normalization shapes (rows of 384 and 8192
# elements, a 1280-wide fp16 case) with attention-logit-like inputs,
# x = x_std * N(0, 1), and optionally a fraction of positions masked to -inf.

@dataclass(frozen=True)
class SoftmaxWorkload:
    name: str
    dtype: str
    rows: int
    hidden: int
    x_std: float = 2.0
    mask_frac: float = 0.0        # positions set to -inf (distinct, uniform)
    masked_rows: int = 0          # whole rows set to -inf (the first ones drawn)

    def with_(self, **kw) -> "SoftmaxWorkload":
        return replace(self, **kw)


SMX_F32_4096x384 = SoftmaxWorkload(name="softmax_f32_4096x384", dtype="f32", rows=4096,
                                   hidden=384)
SMX_F16_8192x1280_MASKED = SoftmaxWorkload(name="softmax_f16_8192x1280_masked", dtype="f16",
                                           rows=8192, hidden=1280, mask_frac=0.25,
                                           masked_rows=3)
SMX_BF16_576000x384 = SoftmaxWorkload(name="softmax_bf16_576000x384", dtype="bf16",
                                      rows=576000, hidden=384)
SMX_BF16_16384x8192 = SoftmaxWorkload(name="softmax_bf16_16384x8192", dtype="bf16",
                                      rows=16384, hidden=8192)

SOFTMAX_WORKLOADS = {w.name: w for w in (SMX_F32_4096x384, SMX_F16_8192x1280_MASKED,
                                         SMX_BF16_576000x384, SMX_BF16_16384x8192)}


def make_softmax_inputs(w: SoftmaxWorkload, seed: int = 0) -> torch.Tensor:
    """x for a softmax workload: draws in the order x, masked positions,
    masked rows; float64 -> float32 -> dtype as for the normalization."""
    rng = np.random.Generator(np.random.PCG64(seed))
    R, H = w.rows, w.hidden
    x = w.x_std * rng.standard_normal((R, H))
    if w.mask_frac > 0.0 and R * H > 0:
        k = int(round(w.mask_frac * R * H))
        x.reshape(-1)[rng.choice(R * H, size=k, replace=False)] = -np.inf
    if w.masked_rows > 0 and R > 0:
        x[rng.choice(R, size=min(R, w.masked_rows), replace=False)] = -np.inf
    return to_dtype(x, w.dtype)


def as_f64(t) -> np.ndarray | None:
    """Decode a CPU tensor of any of the I/O dtypes to a float64 numpy array."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()
