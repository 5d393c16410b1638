"""Benchmark of the fused normalization block (forward + backward step).

One step is the whole hot path on one batch: ln_fwd (bias + residual add,
LayerNorm, amax) followed by ln_bwd (dx, dgamma, dbeta) on the 576000 x 384
bf16 workload. Inputs (442 MB per [rows, hidden] tensor) are larger than L2,
so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu-baseline] [--no-clocks]

``--workload rms_fwd_bwd_bf16_16384x8192`` or
``ln_fwd_bwd_fp8_dbias_bf16_576000x384`` time other forward + backward steps
(the default line also carries the first under ``workloads``);
``softmax_bf16_576000x384`` / ``softmax_bf16_16384x8192`` time the row softmax
(ln_softmax_fwd) and ``partials_bf16_576000x384`` the normalize-from-partials
step (ln_fwd_from_partials), each with its own metric line. The other
configurations the block is checked on have lines of their own too:
``ln_f32_4096x384`` (fwd + bwd), ``bwd_ln_bf16_576000x384`` and
``bwd_rms_bf16_576000x384`` (the backward alone), ``fwd_amax_bf16_32768x768``
(the forward alone) and ``unet_ln_f16_8192x{320,640,1280}`` (fwd + bwd);
those whose buffers fit in L2 cycle through enough copies of them that no
step reads its inputs from L2.

Rank 0 prints one JSON line. Under torchrun (N > 1) every rank runs its own
replica of the workload on its own GPU (the block has no cross-row exchange),
timing is bracketed by barriers and the max over ranks is reported.
``--impl reference`` times the fp64 CPU oracle instead, on host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "fwd+bwd rows/s and achieved HBM GB/s vs ~8 TB/s peak at (576000×384) bf16"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
BENCH_WORKLOADS = {w.name: w for w in (W.BENCH_LN_BF16_576000x384, W.BENCH_RMS_BF16_16384x8192,
                                        W.BENCH_LN_FP8_DBIAS_BF16_576000x384)}
# The normalize-from-partials step is measured on its own workload (its own
# metric line, like the softmax).
PARTIALS_METRIC = ("normalize-from-partials rows/s and achieved HBM GB/s (one read of x and the "
                   "partials, one write of y and the statistics)")
PARTIALS_WORKLOADS = {W.PARTIALS_BF16_576000x384.name: W.PARTIALS_BF16_576000x384}
# The row softmax is measured on its own workloads (its own metric line).
SOFTMAX_METRIC = "softmax rows/s and achieved HBM GB/s (one read of x, one write of y)"
SOFTMAX_WORKLOADS = {w.name: w for w in (W.SMX_BF16_576000x384, W.SMX_BF16_16384x8192)}
# The other configurations the block is checked on, each timed on its own
# line: the fp32 4096 x 384 LayerNorm step, the 576000 x 384 backward alone
# (LayerNorm and RMSNorm, no residual; its statistics come from one untimed
# forward), the 32768 x 768 fused add + LayerNorm + amax forward alone, and
# the three fp16 UNet widths. Buffers that fit in L2 are rotated
# (rotation_copies), so every timed step reads its inputs from HBM.
CONFIG_METRIC = ("rows/s and achieved HBM GB/s of one configuration's calls (forward, backward "
                 "or both)")
CONFIG_WORKLOADS = {w.name: w for w in (W.LN_F32_4096x384, W.BWD_BF16_576000x384_LN,
                                        W.BWD_BF16_576000x384_RMS, W.FWD_AMAX_BF16_32768x768,
                                        *W.UNET_F16.values())}
L2_BYTES_FALLBACK = 129_000_000


def is_softmax(w) -> bool:
    return isinstance(w, W.SoftmaxWorkload)


# ---------------------------------------------------------------- bytes model
def elem_bytes(w) -> int:
    return 4 if w.dtype == "f32" else 2


def fwd_bytes(w) -> int:
    """Minimal HBM bytes of one ln_fwd: each input read once, each output
    written once (x, residual, bias, gamma, beta in; sum, y, stats, amax out;
    with an FP8 copy of y, its R * H bytes and the 4-byte scale)."""
    R, H, e = w.rows, w.hidden, elem_bytes(w)
    has_res = w.residual_std is not None
    store_sum = has_res or w.bias_std is not None
    nstats = 2 if w.mode == W.LAYERNORM else 1
    nparams = 1 + (w.mode == W.LAYERNORM and w.beta_std is not None) + (w.bias_std is not None)
    fp8 = (R * H + 4) if w.fp8_out else 0
    return (R * H * e * (1 + has_res) + R * H * e * (1 + store_sum) + R * 4 * nstats
            + H * e * nparams + (4 if w.amax else 0) + fp8)


def bwd_bytes(w) -> int:
    """Minimal HBM bytes of one ln_bwd: dy, x_sum, stats, gamma in; dx,
    dgamma (and dbeta) out. The workspace partials are not counted."""
    R, H, e = w.rows, w.hidden, elem_bytes(w)
    nstats = 2 if w.mode == W.LAYERNORM else 1
    ngrads = (2 if w.mode == W.LAYERNORM else 1) + (1 if w.dbias else 0)
    return 3 * R * H * e + R * 4 * nstats + H * e + H * 4 * ngrads


def partials_bytes(w, tile_cols) -> int:
    """Minimal HBM bytes of one ln_fwd_from_partials: x and the two fp32
    partials per tile read once; y, the statistics and amax written once."""
    R, H, e = w.rows, w.hidden, elem_bytes(w)
    T = -(-H // tile_cols)
    nstats = 2 if w.mode == W.LAYERNORM else 1
    nparams = 1 + (w.mode == W.LAYERNORM and w.beta_std is not None)
    return (2 * R * H * e + R * T * 8 + R * 4 * nstats + H * e * nparams
            + (4 if w.amax else 0))


def softmax_bytes(w) -> int:
    """Minimal HBM bytes of one ln_softmax_fwd: x read once, y written once."""
    return 2 * w.rows * w.hidden * elem_bytes(w)


def step_bytes(w) -> int:
    """Minimal HBM bytes of one timed step: the calls the workload makes."""
    return (fwd_bytes(w) if w.forward else 0) + (bwd_bytes(w) if w.backward else 0)


def rotation_copies(w, l2_bytes: int) -> int:
    """Buffer sets a timed loop cycles through: one when every [rows, hidden]
    tensor is larger than L2; otherwise enough sets that a pass over them
    moves at least three times the L2's bytes, so the inputs a step reads
    were last touched three L2s of traffic earlier (evicted, not L2 hits)."""
    if w.rows * w.hidden * elem_bytes(w) > l2_bytes:
        return 1
    return max(2, -(-3 * l2_bytes // step_bytes(w)))


def l2_bytes(device) -> int:
    props = torch.cuda.get_device_properties(device)
    return int(getattr(props, "L2_cache_size", 0) or L2_BYTES_FALLBACK)


# ---------------------------------------------------------------- clocks
_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown"}


class ClockSampler:
    """Samples the GPU's SM clock, power and clock-event reasons in a
    background thread while the workload runs.

    Reads NVML directly through ctypes (libnvidia-ml ships with the driver;
    only read-only queries are made) every ``period_s`` (2 ms), so even a
    timed region of a few milliseconds gets samples; falls back to
    ``nvidia-smi -lms 10`` when NVML cannot be loaded."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.samples = []       # (time, sm_mhz, sm_max_mhz, power_w, [reasons])
        self.proc = None
        self.source = None
        self._stop = threading.Event()
        uuid = None
        try:
            u = getattr(torch.cuda.get_device_properties(device_index), "uuid", None)
            uuid = ("GPU-" + str(u)) if u else None
        except Exception:
            pass
        if self._nvml_open(uuid):
            self.source = f"nvml every {period_s * 1e3:.0f} ms"
            self.thread = threading.Thread(target=self._poll_nvml, args=(period_s,), daemon=True)
            self.thread.start()
        else:
            self._smi_open(uuid)

    # -- NVML
    def _nvml_open(self, uuid) -> bool:
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            if uuid is not None:
                if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                    return False
            elif lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                return False
            self._nvml, self._h, self._ct = lib, h, ctypes
            mx = ctypes.c_uint(0)
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))      # 1 = NVML_CLOCK_SM
            self._max = float(mx.value) or None
            self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            return True
        except (OSError, AttributeError):
            return False

    def _poll_nvml(self, period_s):
        ct, lib, h = self._ct, self._nvml, self._h
        clk, pw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        while not self._stop.is_set():
            t = time.time()
            ok = lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0
            p = float(pw.value) / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ct.byref(pw)) == 0 \
                else None
            r = int(rs.value) if self._reasons_fn(h, ct.byref(rs)) == 0 else 0
            if ok:
                self.samples.append((t, float(clk.value), self._max, p,
                                     [n for b, n in _REASONS.items() if r & b]))
            self._stop.wait(period_s)

    # -- nvidia-smi fallback
    def _smi_open(self, uuid):
        for gid in ([uuid] if uuid else []) + [None]:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "10"]
            if gid:
                cmd += ["-i", gid]
            try:
                p = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                     text=True)
            except OSError:
                return
            time.sleep(0.3)
            if p.poll() is None:
                self.proc = p
                self.source = "nvidia-smi -lms 10"
                break
        if self.proc is not None:
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9 and num(parts[1]) is not None:
                self.samples.append((time.time(), num(parts[1]), num(parts[2]), num(parts[3]),
                                     [n for n, v in zip(names, parts[5:9])
                                      if v.lower() == "active"]))

    def stop(self):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float, window: str):
        win = [x for x in self.samples if t0 <= x[0] <= t1]
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": len(win),
               "window": window, "source": self.source}
        if not win:
            return out
        sm = [x[1] for x in win]
        smax = [x[2] for x in win if x[2] is not None]
        power = [x[3] for x in win if x[3] is not None]
        out.update({"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm),
                    "sm_max_mhz": max(smax) if smax else None,
                    "reasons": sorted({r for x in win for r in x[4]}),
                    "power_w_max": max(power) if power else None})
        return out


# ---------------------------------------------------------------- helpers
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Host-side sources (planning, argument checks, entry points) do not change
# what a kernel reads or writes, so they are left out of the kernel hash.
HOST_SOURCES = ("api.cu", "plan.cu", "noalloc.cu", "launch.h")


def source_hash() -> str:
    """Hash of the kernel sources the committed ncu traffic was taken from."""
    d = os.path.join(ROOT, "normalization_fwd_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh")) and name not in HOST_SOURCES:
            with open(os.path.join(d, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_hash") != source_hash():
        return None
    return d.get("workloads", {}).get(workload, {}).get(kernel)


class Step:
    """Device buffers and the C-ABI calls of one step: ln_fwd then ln_bwd,
    or only the one the workload has (w.forward / w.backward). A backward-only
    workload (no bias, no residual: the backward's x_sum is x itself) gets
    its statistics from one untimed ln_fwd here, as inputs."""

    def __init__(self, nf, w, inp, device):
        self.nf, self.w = nf, w
        g = {k: (v.to(device) if v is not None else None) for k, v in inp.items()}
        self.inp = g
        R, H = w.rows, w.hidden
        dt = W.TORCH_DTYPES[w.dtype]
        self.rms = w.mode == W.RMSNORM
        f32 = dict(dtype=torch.float32, device=device)
        if not w.forward and (w.bias_std is not None or w.residual_std is not None):
            raise ValueError(f"{w.name}: a backward-only step takes x as its sum (no add)")
        self.sum = torch.empty(R, H, dtype=dt, device=device) if w.forward else g["x"]
        self.y = torch.empty(R, H, dtype=dt, device=device) if w.forward else None
        self.mean = None if self.rms else torch.empty(R, **f32)
        self.rstd = torch.empty(R, **f32)
        self.amax = torch.empty(1, **f32) if (w.amax and w.forward) else None
        bwd = w.backward
        self.dx = torch.empty(R, H, dtype=dt, device=device) if bwd else None
        self.dgamma = torch.empty(H, **f32) if bwd else None
        self.dbeta = None if (self.rms or not bwd) else torch.empty(H, **f32)
        self.dbias = torch.empty(H, **f32) if (w.dbias and bwd) else None
        # FP8 copy of y with a per-tensor scale (delayed scaling: 448 over an
        # amax of an earlier step; a fixed value here)
        self.y_fp8 = torch.empty(R, H, dtype=torch.uint8, device=device) if w.fp8_out else None
        self.fp8_scale = torch.full((1,), 64.0, **f32) if w.fp8_out else None
        self.ws = None
        if bwd:
            need = nf.ln_bwd_workspace_bytes(R, H, dt, w.mode)
            self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        if not w.forward:
            y = torch.empty(R, H, dtype=dt, device=device)
            nf.ln_fwd(g["x"], None, None, g["gamma"], g["beta"], w.eps, w.mode,
                      w.zero_centered_gamma, None, y, self.mean, self.rstd, None)
            torch.cuda.synchronize(device)
            del y

    def fwd(self, stream):
        g, w = self.inp, self.w
        if not w.forward:
            return
        if w.fp8_out:
            self.nf.ln_fwd_ex(g["x"], g["bias"], g["residual"], g["gamma"], g["beta"], w.eps,
                              w.mode, w.zero_centered_gamma, self.sum, self.y, self.mean,
                              self.rstd, self.amax, self.y_fp8, self.fp8_scale, stream)
            return
        self.nf.ln_fwd(g["x"], g["bias"], g["residual"], g["gamma"], g["beta"], w.eps, w.mode,
                       w.zero_centered_gamma, self.sum, self.y, self.mean, self.rstd, self.amax,
                       stream)

    def bwd(self, stream):
        g, w = self.inp, self.w
        if not w.backward:
            return
        if w.dbias:
            self.nf.ln_bwd_ex(g["dy"], self.sum, g["gamma"], self.mean, self.rstd, self.dx,
                              self.dgamma, self.dbeta, self.dbias, stream, mode=w.mode,
                              zero_centered_gamma=w.zero_centered_gamma, workspace=self.ws)
            return
        self.nf.ln_bwd(g["dy"], self.sum, g["gamma"], self.mean, self.rstd, self.dx, self.dgamma,
                       self.dbeta, stream, mode=w.mode, zero_centered_gamma=w.zero_centered_gamma,
                       workspace=self.ws)

    def run(self, stream):
        self.fwd(stream)
        self.bwd(stream)

    def h2d_tensors(self):
        ins = [(k, self.inp[k]) for k in ("x", "residual", "bias", "gamma", "beta", "dy")
               if self.inp[k] is not None]
        if not self.w.forward:   # the statistics are inputs of a backward-only step
            ins += [(k, t) for k, t in (("mean", self.mean), ("rstd", self.rstd))
                    if t is not None]
        return ins

    def d2h_tensors(self):
        out = [("dx", self.dx), ("dgamma", self.dgamma), ("dbeta", self.dbeta),
               ("dbias", self.dbias)]
        if self.w.forward:
            out = [("sum", self.sum), ("y", self.y), ("mean", self.mean), ("rstd", self.rstd),
                   ("amax", self.amax), ("y_fp8", self.y_fp8)] + out
        return [(k, t) for k, t in out if t is not None]

    def launches(self) -> int:
        """Kernels of this library one step launches (the backward's main
        kernel and its finalize)."""
        return (1 if self.w.forward else 0) + (2 if self.w.backward else 0)


class RotatingStep:
    """`copies` Steps over their own buffers, used in turn (step i on set
    i mod copies), so buffers that would fit in L2 are not re-read from it."""

    def __init__(self, nf, w, inp, device, copies):
        self.steps = [Step(nf, w, inp, device) for _ in range(copies)]
        self.i = 0

    def fwd(self, stream):
        self.steps[self.i].fwd(stream)

    def bwd(self, stream):
        self.steps[self.i].bwd(stream)
        self.i = (self.i + 1) % len(self.steps)

    def launches(self) -> int:
        return self.steps[0].launches()


def producer_partials(x, tile_cols):
    """Stand-in for the producer of the partials (a GEMM epilogue, outside
    this library): per row and column tile, the fp32 sum and sum of squares
    of the stored row, taken with torch on the device as input data."""
    R, H = x.shape
    T = -(-H // tile_cols)
    xf = torch.nn.functional.pad(x.float(), (0, T * tile_cols - H)).view(R, T, tile_cols)
    return xf.sum(-1).contiguous(), (xf * xf).sum(-1).contiguous()


def make_partials_inputs(w, seed=0):
    """The workload's x, gamma, beta and the producer stand-in's partials
    (computed on the host in 65536-row blocks)."""
    inp = W.make_inputs(w, seed=seed)
    parts = [producer_partials(inp["x"][i:i + 65536], W.PARTIALS_TILE_COLS)
             for i in range(0, w.rows, 65536)]
    inp["psum"] = torch.cat([p[0] for p in parts])
    inp["psq"] = torch.cat([p[1] for p in parts])
    return inp


class PartialsStep:
    """Device buffers and the C-ABI call of one normalize-from-partials step."""

    def __init__(self, nf, w, inp_host, device):
        self.nf, self.w = nf, w
        self.tile = W.PARTIALS_TILE_COLS
        self.x = inp_host["x"].to(device)
        self.gamma = inp_host["gamma"].to(device)
        self.beta = inp_host["beta"].to(device) if inp_host["beta"] is not None else None
        self.psum = inp_host["psum"].to(device)
        self.psq = inp_host["psq"].to(device)
        R = w.rows
        f32 = dict(dtype=torch.float32, device=device)
        self.y = torch.empty_like(self.x)
        self.mean = None if w.mode == W.RMSNORM else torch.empty(R, **f32)
        self.rstd = torch.empty(R, **f32)
        self.amax = torch.empty(1, **f32) if w.amax else None

    def run(self, stream):
        w = self.w
        self.nf.ln_fwd_from_partials(self.x, self.psum, self.psq, self.tile, "sum_sq", self.gamma,
                                     self.beta, w.eps, w.mode, w.zero_centered_gamma, self.y,
                                     self.mean, self.rstd, self.amax, stream)

    def h2d_tensors(self):
        return [("x", self.x), ("psum", self.psum), ("psq", self.psq)]

    def d2h_tensors(self):
        out = [("y", self.y), ("mean", self.mean), ("rstd", self.rstd), ("amax", self.amax)]
        return [(k, t) for k, t in out if t is not None]


class SoftmaxStep:
    """Device buffers and the C-ABI call of one row softmax step."""

    def __init__(self, nf, w, x_host, device):
        self.nf, self.w = nf, w
        self.x = x_host.to(device)
        self.y = torch.empty_like(self.x)

    def run(self, stream):
        self.nf.ln_softmax_fwd(self.x, self.y, stream)

    def h2d_tensors(self):
        return [("x", self.x)]

    def d2h_tensors(self):
        return [("y", self.y)]


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The max of a per-rank timing over all ranks (all_reduce MAX); the
    value itself when running alone. Works with NCCL (CUDA tensor) and gloo
    (CPU tensor)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(rows_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job rows/s of `world` replicas, each stepping `rows_per_rank`
    rows in `ms_per_step` (the slowest rank's time)."""
    return world * rows_per_rank / (ms_per_step * 1e-3)


def nbytes(t) -> int:
    return t.numel() * t.element_size()


# ---------------------------------------------------------------- oracle timing
def oracle_step(w, inp, rows):
    """One step of the fp64 oracle over the first `rows` rows: forward, then
    backward (a backward-only workload takes its statistics from the
    oracle's forward, inside the step; a forward-only one stops there)."""
    from oracle import norm_bwd, norm_fwd
    sl = slice(0, rows)
    f = W.as_f64
    res = inp["residual"]
    ref = norm_fwd(f(inp["x"][sl]), f(inp["bias"]), None if res is None else f(res[sl]),
                   f(inp["gamma"]), f(inp["beta"]), w.eps, w.mode, w.zero_centered_gamma,
                   w.dtype)
    if w.backward:
        norm_bwd(f(inp["dy"][sl]), ref["sum"], f(inp["gamma"]), ref["mean"], ref["rstd"],
                 w.mode, w.zero_centered_gamma, w.dtype)


def oracle_what(w) -> str:
    if w.forward and w.backward:
        return "fwd+bwd"
    if w.forward:
        return "fwd"
    return "bwd (with the forward for its statistics)"


def oracle_softmax_step(w, x, rows):
    """One fp64 oracle softmax over the first `rows` rows."""
    from oracle import softmax_fwd
    softmax_fwd(W.as_f64(x[:rows]), w.dtype)


def oracle_partials_step(w, inp, rows):
    """One fp64 oracle normalize-from-partials over the first `rows` rows."""
    from oracle import norm_fwd_from_partials
    f = W.as_f64
    norm_fwd_from_partials(f(inp["x"][:rows]), f(inp["psum"][:rows]), f(inp["psq"][:rows]),
                           W.PARTIALS_TILE_COLS, "sum_sq", f(inp["gamma"]), f(inp["beta"]), w.eps,
                           w.mode, w.zero_centered_gamma, w.dtype)


def is_partials(w) -> bool:
    return w.name.split("@")[0] in PARTIALS_WORKLOADS


def oracle_any_step(w, inp, rows):
    if is_softmax(w):
        oracle_softmax_step(w, inp, rows)
    elif is_partials(w):
        oracle_partials_step(w, inp, rows)
    else:
        oracle_step(w, inp, rows)


def time_oracle(w, inp, budget_s: float):
    """rows/s of the oracle on a sample sized to about `budget_s` of CPU work."""
    probe = min(2048, w.rows)
    t0 = time.perf_counter()
    oracle_any_step(w, inp, probe)
    t_probe = time.perf_counter() - t0
    rows = int(min(w.rows, max(probe, probe * budget_s / max(t_probe, 1e-6))))
    rows = min(rows, 131072)
    t0 = time.perf_counter()
    oracle_any_step(w, inp, rows)
    dt = time.perf_counter() - t0
    return rows / dt, rows, dt


def _oracle_worker(args):
    """One host process of the all-cores oracle timing: draw a same-shape
    sample of the workload (its own seed; the oracle's speed does not depend
    on the values), wait for every worker, then time the oracle on it."""
    w, rows, seed, barrier = args
    import time as _t
    smx = isinstance(w, W.SoftmaxWorkload)
    sample = w.with_(rows=rows)
    if smx:
        inp = W.make_softmax_inputs(sample, seed=seed)
    elif is_partials(w):
        inp = make_partials_inputs(sample, seed=seed)
    else:
        inp = W.make_inputs(sample, seed=seed)
    barrier.wait()
    t0 = _t.perf_counter()
    oracle_any_step(sample, inp, rows)
    return rows, _t.perf_counter() - t0


def time_oracle_all_cores(w, rows_per_worker: int, procs: int):
    """rows/s of the oracle run by `procs` host processes at once (a spawn
    pool, so no CUDA state is inherited; numpy single-threaded in each)."""
    import multiprocessing as mp
    env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in env_keys}
    for k in env_keys:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Manager() as mgr:
            barrier = mgr.Barrier(procs)
            with ctx.Pool(procs) as pool:
                res = pool.map(_oracle_worker,
                               [(w, rows_per_worker, 100 + i, barrier) for i in range(procs)])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    rows = sum(r for r, _ in res)
    secs = max(t for _, t in res)
    return rows / secs, rows, secs


def cpu_baselines(w, inp_host, what):
    """The oracle on one host core (the contract's cpu_baseline) and on all
    of them (one process per core)."""
    v, rows, secs = time_oracle(w, inp_host, budget_s=12.0)
    one = {"value": v, "unit": "rows/s", "cores": 1, "kind": "oracle",
           "sample": f"first {rows} of {w.rows} rows, fp64 numpy oracle {what}, "
                     f"{secs:.1f} s on 1 host thread"}
    procs = max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                else (os.cpu_count() or 1))
    # about 4 s of oracle work per process, at most 4 Mi elements per tensor
    # (host memory: every process holds its own sample)
    per = int(rows * 4.0 / max(secs, 1e-6))
    per = max(16, min(per, rows, (4 << 20) // w.hidden))
    va, rows_a, secs_a = time_oracle_all_cores(w, per, procs)
    allc = {"value": va, "unit": "rows/s", "cores": procs, "kind": "oracle",
            "sample": f"{procs} processes x {per} rows (same shape and distribution, own "
                      f"seeds), fp64 numpy oracle {what}, {secs_a:.1f} s wall"}
    return one, allc


# ---------------------------------------------------------------- arms
def run_reference(args, w, rank):
    """The oracle on host cores, as the reference arm."""
    if rank != 0:
        return
    smx = is_softmax(w)
    if smx:
        inp = W.make_softmax_inputs(w, seed=0)
    elif is_partials(w):
        inp = make_partials_inputs(w, seed=0)
    else:
        inp = W.make_inputs(w, seed=0)
    budget = 60.0   # seconds of oracle work over all steps of the arm
    probe = min(1024, w.rows)
    t0 = time.perf_counter()
    oracle_any_step(w, inp, probe)
    per_row = (time.perf_counter() - t0) / probe
    steps = args.steps + args.warmup
    rows = max(16, min(w.rows, int(budget / max(steps, 1) / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        oracle_any_step(w, inp, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_any_step(w, inp, rows)
    el = time.perf_counter() - t0
    value = rows * args.steps / el
    what = "softmax" if smx else ("normalize from partials" if is_partials(w) else oracle_what(w))
    sample = f"first {rows} of {w.rows} rows per step, fp64 numpy oracle {what}, 1 thread"
    ms_step = 1000.0 * el / args.steps
    line = {
        "impl": "reference", "metric": metric_of(w), "value": value,
        "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # measured: one step is the oracle over the sampled rows
        "ms_per_step": ms_step, "rows_per_step": rows,
        # what a step over every row of the workload would take at that rate
        "ms_per_step_full_rows_extrapolated": ms_step * (w.rows / rows),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def is_config(w) -> bool:
    return w.name.split("@")[0] in CONFIG_WORKLOADS


def metric_of(w):
    if is_softmax(w):
        return SOFTMAX_METRIC
    if is_partials(w):
        return PARTIALS_METRIC
    if is_config(w):
        return CONFIG_METRIC
    return METRIC


def config_of(w, n, copies=1):
    if is_softmax(w):
        return {"workload": w.name, "rows": w.rows, "hidden": w.hidden, "io_dtype": w.dtype,
                "x_std": w.x_std, "mask_frac": w.mask_frac,
                "l2": "no flush: x and y are each larger than the 129 MB L2",
                "parallelism": "replicas" if n > 1 else "single-gpu"}
    c = {"workload": w.name, "rows": w.rows, "hidden": w.hidden, "mode": w.mode,
         "io_dtype": w.dtype, "stats_dtype": "f32", "bias": w.bias_std is not None,
         "residual": w.residual_std is not None, "amax": w.amax, "eps": w.eps,
         "l2": "no flush: every [rows, hidden] input is larger than the 129 MB L2",
         "parallelism": "replicas" if n > 1 else "single-gpu"}
    if w.fp8_out:
        c["fp8_out"] = "E4M3 copy of y, per-tensor scale"
    if w.dbias:
        c["dbias"] = True
    if is_partials(w):
        c["partials"] = {"kind": "sum_sq", "tile_cols": W.PARTIALS_TILE_COLS,
                         "producer": "fp32 tile sums of the stored row, precomputed (stand-in)"}
    if is_config(w):
        c["calls"] = [k for k, on in (("ln_fwd", w.forward), ("ln_bwd", w.backward)) if on]
        if not w.forward:
            c["stats"] = "mean/rstd from one untimed ln_fwd of x (inputs of the backward)"
        if w.zero_centered_gamma:
            c["zero_centered_gamma"] = True
    if copies > 1:
        c["l2"] = (f"no flush: the steps cycle through {copies} copies of every buffer "
                   f"({copies} x {step_bytes(w)} algorithmic bytes, at least 3x the L2), so "
                   "each step reads inputs last touched 3 L2s of traffic earlier")
        c["timing"] = ("the K steps captured in one CUDA graph and replayed (per-call means "
                       "from graphs of K forwards and K backwards)")
    return c


def clock_record(sampler, t_warm0, t_host0, t_host1):
    """The clock samples of the timed region; when it is too short for a few
    samples (a few ms at --steps 20), those of the warm-up plus the timed
    region, which run the same kernels back to back. Both are kept."""
    if sampler is None:
        return None
    time.sleep(0.01)   # let the sampler thread append the samples it is taking
    timed = sampler.summary(t_host0, t_host1, "timed")
    rec = timed if timed["samples"] >= 3 else sampler.summary(t_warm0, t_host1, "warmup+timed")
    rec = dict(rec)
    rec["timed_region"] = timed
    return rec


def time_fwd_bwd(nf, w, inp_host, device, args, world, sampler, copies=1):
    """Warm up, then time exactly K fused steps (ln_fwd + ln_bwd, or the one
    call the workload has) between barriers with CUDA events on the launching
    stream; per-kernel means from events around each call. copies > 1: the
    steps cycle through that many buffer sets (RotatingStep)."""
    step = (RotatingStep(nf, w, inp_host, device, copies) if copies > 1
            else Step(nf, w, inp_host, device))
    launches = step.launches()
    stream = torch.cuda.current_stream(device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    torch.cuda.synchronize(device)
    t_warm0 = time.time()
    for _ in range(args.warmup):
        step.fwd(stream)
        step.bwd(stream)
    torch.cuda.synchronize(device)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(device)
    t_host0 = time.time()
    start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        step.fwd(stream)
        ev[i][1].record(stream)
        step.bwd(stream)
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize(device)
    t_host1 = time.time()
    barrier()
    elapsed = max_over_ranks(start.elapsed_time(end), world, device)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    del step
    torch.cuda.empty_cache()
    return {"ms_step": elapsed / K, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "launches_per_step": launches,
            "clocks": clock_record(sampler, t_warm0, t_host0, t_host1)}


def time_fwd_bwd_graph(nf, w, inp_host, device, args, world, sampler, copies):
    """The configurations whose buffers fit in L2: their calls take 6-40 us,
    about what the host needs to issue a call through Python and ctypes, so
    an eager loop would time the host. The K timed steps (cycling through `copies` buffer
    sets) are captured into one CUDA graph and replayed once between
    barriers, with CUDA events around the replay; for a forward + backward
    step, K forwards alone and K backwards alone are captured and replayed
    the same way for the per-call means."""
    step = RotatingStep(nf, w, inp_host, device, copies)
    launches = step.launches()
    n = len(step.steps)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    torch.cuda.synchronize(device)
    t_warm0 = time.time()
    with torch.cuda.stream(side):   # eager warm-up: plans and kernel attributes
        for _ in range(args.warmup):
            step.fwd(side)
            step.bwd(side)
    torch.cuda.synchronize(device)

    K = args.steps

    def capture(do_fwd, do_bwd):
        g = torch.cuda.CUDAGraph()
        step.i = 0
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream(device)
            for _ in range(K):
                if do_fwd:
                    step.steps[step.i].fwd(cs)
                if do_bwd:
                    step.steps[step.i].bwd(cs)
                step.i = (step.i + 1) % n
        return g

    graphs = {"step": capture(True, True)}
    if w.forward and w.backward:
        graphs["fwd"] = capture(True, False)
        graphs["bwd"] = capture(False, True)
    stream = torch.cuda.current_stream(device)
    times = {"fwd": 0.0, "bwd": 0.0}
    t_host0 = t_host1 = None
    for name in [k for k in ("fwd", "bwd") if k in graphs] + ["step"]:
        g = graphs[name]
        g.replay()                      # warm replay
        torch.cuda.synchronize(device)
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize(device)
        h0 = time.time()
        a.record(stream)
        g.replay()
        z.record(stream)
        torch.cuda.synchronize(device)
        h1 = time.time()
        barrier()
        times[name] = max_over_ranks(a.elapsed_time(z), world, device)
        if name == "step":
            t_host0, t_host1 = h0, h1
    if not (w.forward and w.backward):   # one call per step: the step is that call
        times["fwd" if w.forward else "bwd"] = times["step"]
    del graphs, step
    torch.cuda.empty_cache()
    return {"ms_step": times["step"] / K, "fwd_ms": times["fwd"] / K,
            "bwd_ms": times["bwd"] / K, "launches_per_step": launches,
            "clocks": clock_record(sampler, t_warm0, t_host0, t_host1)}


def kernel_report(w, t):
    """Per-kernel algorithmic GB/s against the measured copy peak and the
    nominal 8 TB/s, and the roofline of the dominant kernel."""
    peak, peak_kind = measured_peak()
    fb = fwd_bytes(w) if w.forward else 0
    bb = bwd_bytes(w) if w.backward else 0
    calls = [c for c, on in ((("ln_fwd", t["fwd_ms"], fb), w.forward),
                             (("ln_bwd", t["bwd_ms"], bb), w.backward)) if on]
    kernels = {}
    for name, ms, by in calls:
        gbs = by / (ms * 1e-3) / 1e9
        kernels[name] = {"us": ms * 1e3, "algorithmic_bytes": by, "GBps": gbs,
                         f"frac_of_{peak_kind}": gbs / peak, "frac_of_8TBps": gbs / NOMINAL_HBM_GBS,
                         "traffic": ncu_traffic(w.name, name)}
    dom = max(kernels, key=lambda k: kernels[k]["us"])
    d = kernels[dom]
    roofline = {"bound": "hbm", "kernel": dom, "achieved": d["GBps"], "peak": peak,
                "unit": "GB/s", "frac": d["GBps"] / peak, "peak_kind": peak_kind,
                "traffic": d["traffic"]}
    return kernels, roofline, (fb + bb) / (t["ms_step"] * 1e-3) / 1e9


# The second shape the HBM target is stated at: timed in the same run as the
# default workload and reported under "workloads" on the same line.
SECOND_GATE_WORKLOAD = W.BENCH_RMS_BF16_16384x8192


def run_ours(args, w, rank, world, local_rank):
    import normalization_fwd_gb300 as nf
    nf.load_library()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    inp_host = W.make_inputs(w, seed=0)
    copies = rotation_copies(w, l2_bytes(device))
    sampler = ClockSampler(local_rank) if (rank == 0 and not args.no_clocks) else None
    if sampler is not None:
        time.sleep(0.3)
    if copies > 1:
        t = time_fwd_bwd_graph(nf, w, inp_host, device, args, world, sampler, copies)
    else:
        t = time_fwd_bwd(nf, w, inp_host, device, args, world, sampler)

    # the second gate shape, same steps and warm-up (default workload only)
    extra = {}
    second = (not args.no_second and args.rows is None
              and w.name == W.BENCH_LN_BF16_576000x384.name)
    if second:
        w2 = SECOND_GATE_WORKLOAD
        t2 = time_fwd_bwd(nf, w2, W.make_inputs(w2, seed=0), device, args, world, sampler)
        k2, r2, g2 = kernel_report(w2, t2)
        extra[w2.name] = {
            "value": replica_throughput(w2.rows, world, t2["ms_step"]), "unit": "rows/s",
            "ms_per_step": t2["ms_step"], "config": config_of(w2, world), "roofline": r2,
            "kernels": k2, "step_GBps": g2, "gpu_launches": t2["launches_per_step"] * args.steps,
            "clocks": t2["clocks"]}
    if sampler is not None:
        time.sleep(0.05)
        sampler.stop()

    # end to end through the same calls, inputs from pinned host memory and
    # every output read back, each step
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(nf, w, inp_host, device, min(args.e2e_steps, max(args.steps, 1)))

    if rank != 0:
        return
    kernels, roofline, step_gbs = kernel_report(w, t)
    cpu = cpu_all = None
    if not args.no_cpu_baseline and world == 1:
        cpu, cpu_all = cpu_baselines(w, inp_host, oracle_what(w))
    K = args.steps
    line = {
        "metric": metric_of(w), "value": replica_throughput(w.rows, world, t["ms_step"]),
        "unit": "rows/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": t["ms_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_of(w, world, copies),
        "roofline": roofline, "kernels": kernels, "step_GBps": step_gbs,
        "cpu_baseline": cpu, "cpu_baseline_all_cores": cpu_all, "e2e": e2e,
        "gpu_launches": t["launches_per_step"] * K, "clocks": t["clocks"], "impl": "ours",
    }
    if extra:
        line["workloads"] = extra
    print(json.dumps(line), flush=True)


def run_softmax(args, w, rank, world, local_rank):
    """Time ln_softmax_fwd alone on a softmax workload, or
    ln_fwd_from_partials alone on a partials workload (its own JSON line)."""
    import normalization_fwd_gb300 as nf
    nf.load_library()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    part = is_partials(w)
    x_host = make_partials_inputs(w, seed=0) if part else W.make_softmax_inputs(w, seed=0)
    step_cls = PartialsStep if part else SoftmaxStep
    kname = "ln_fwd_from_partials" if part else "ln_softmax_fwd"
    step = step_cls(nf, w, x_host, device)
    stream = torch.cuda.current_stream(device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    sampler = ClockSampler(local_rank) if (rank == 0 and not args.no_clocks) else None
    if sampler is not None:
        time.sleep(0.3)
    torch.cuda.synchronize(device)
    t_warm0 = time.time()
    for _ in range(args.warmup):
        step.run(stream)
    torch.cuda.synchronize(device)
    K = args.steps
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(device)
    t_host0 = time.time()
    start.record(stream)
    for _ in range(K):
        step.run(stream)
    end.record(stream)
    torch.cuda.synchronize(device)
    t_host1 = time.time()
    barrier()
    elapsed = max_over_ranks(start.elapsed_time(end), world, device)
    clocks = clock_record(sampler, t_warm0, t_host0, t_host1)
    if sampler is not None:
        sampler.stop()
    e2e = None
    if not args.no_e2e:
        del step
        torch.cuda.empty_cache()
        e2e = run_e2e(nf, w, x_host, device, min(args.e2e_steps, max(K, 1)),
                      make_step=step_cls)
    if rank != 0:
        return
    peak, peak_kind = measured_peak()
    ms = elapsed / K
    by = partials_bytes(w, W.PARTIALS_TILE_COLS) if part else softmax_bytes(w)
    gbs = by / (ms * 1e-3) / 1e9
    kernels = {kname: {"us": ms * 1e3, "algorithmic_bytes": by, "GBps": gbs,
                       f"frac_of_{peak_kind}": gbs / peak, "frac_of_8TBps": gbs / NOMINAL_HBM_GBS,
                       "traffic": ncu_traffic(w.name, kname)}}
    roofline = {"bound": "hbm", "kernel": kname, "achieved": gbs, "peak": peak,
                "unit": "GB/s", "frac": gbs / peak, "peak_kind": peak_kind,
                "traffic": kernels[kname]["traffic"]}
    cpu = cpu_all = None
    if not args.no_cpu_baseline and world == 1:
        cpu, cpu_all = cpu_baselines(w, x_host, "normalize from partials" if part else "softmax")
    line = {
        "metric": metric_of(w), "value": replica_throughput(w.rows, world, ms),
        "unit": "rows/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic", "config": config_of(w, world),
        "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all, "e2e": e2e,
        "gpu_launches": K, "clocks": clocks, "impl": "ours",
    }
    print(json.dumps(line), flush=True)


def run_e2e(nf, w, inp_host, device, steps, make_step=Step):
    """The same step end to end from pinned host memory: every step copies
    its inputs host -> device, runs the step's C-ABI calls, and copies every
    output device -> host. Two buffer sets alternate so step i + 1's upload
    (copy stream) overlaps step i's compute (compute stream) and download
    (a third stream); each direction has its own copy engine."""
    sets = [make_step(nf, w, inp_host, device) for _ in range(2)]
    h2d = [s.h2d_tensors() for s in sets]
    d2h = [s.d2h_tensors() for s in sets]
    host_in = {k: t.detach().to("cpu").pin_memory() for k, t in h2d[0]}
    host_out = [{k: torch.empty(t.shape, dtype=t.dtype).pin_memory() for k, t in d} for d in d2h]
    up, comp, down = (torch.cuda.Stream(device) for _ in range(3))
    uploaded = [torch.cuda.Event() for _ in sets]
    computed = [torch.cuda.Event() for _ in sets]
    downloaded = [torch.cuda.Event() for _ in sets]

    def one(i):
        b = i % 2
        if i >= 2:                      # set b is free once its last use is done
            up.wait_event(computed[b])
            up.wait_event(downloaded[b])
        with torch.cuda.stream(up):
            for k, t in h2d[b]:
                t.copy_(host_in[k], non_blocking=True)
            uploaded[b].record(up)
        comp.wait_event(uploaded[b])
        sets[b].run(comp)
        computed[b].record(comp)
        down.wait_event(computed[b])
        with torch.cuda.stream(down):
            for k, t in d2h[b]:
                host_out[b][k].copy_(t, non_blocking=True)
            downloaded[b].record(down)

    for i in range(2):
        one(i)
    torch.cuda.synchronize(device)
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record(up)
    for i in range(steps):
        one(i)
    down.wait_event(computed[(steps - 1) % 2])
    z.record(down)
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(z) / steps
    bi = sum(nbytes(t) for _, t in h2d[0])
    bo = sum(nbytes(t) for _, t in d2h[0])
    # Which side limits: each direction's bytes over the step time, against
    # the copy engines' own rate measured here on one buffer set.
    link = host_link_rates(h2d[0], d2h[0], host_in, host_out[0], device)
    return {"value": w.rows / (ms * 1e-3), "unit": "rows/s", "ms_per_step": ms,
            "steps": steps, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "h2d_GBps": bi / (ms * 1e-3) / 1e9, "d2h_GBps": bo / (ms * 1e-3) / 1e9,
            "host_link": link,
            "pipeline": "2 buffer sets; upload, compute and download on 3 streams"}


def host_link_rates(h2d, d2h, host_in, host_out, device):
    """GB/s of the step's uploads alone and of its downloads alone (pinned
    host memory, one stream each, CUDA events), so the e2e record shows
    whether the step is bound by the host link or by the device."""
    s = torch.cuda.Stream(device)
    out = {}
    for name, pairs in (("h2d_GBps_alone", [(t, host_in[k]) for k, t in h2d]),
                        ("d2h_GBps_alone", [(host_out[k], t) for k, t in d2h])):
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            a.record(s)
            for dst, src in pairs:
                dst.copy_(src, non_blocking=True)
            z.record(s)
        torch.cuda.synchronize(device)
        by = sum(nbytes(d) for d, _ in pairs)
        out[name] = by / (a.elapsed_time(z) * 1e-3) / 1e9
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(BENCH_WORKLOADS) + sorted(SOFTMAX_WORKLOADS)
                    + sorted(PARTIALS_WORKLOADS) + sorted(CONFIG_WORKLOADS),
                    default=W.BENCH_LN_BF16_576000x384.name)
    ap.add_argument("--rows", type=int, default=None,
                    help="override the workload's row count (smaller profiling captures)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-second", action="store_true",
                    help="time only the chosen workload (the default run also times the "
                         "16384 x 8192 RMSNorm step and reports it under 'workloads')")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = (BENCH_WORKLOADS.get(args.workload) or SOFTMAX_WORKLOADS.get(args.workload)
         or PARTIALS_WORKLOADS.get(args.workload) or CONFIG_WORKLOADS[args.workload])
    if args.rows is not None:
        w = w.with_(rows=args.rows, name=f"{w.name}@rows={args.rows}")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world:
        if world == 1 and args.gpus > 1:
            ap.error("--gpus N > 1 runs under torchrun (one process per GPU)")
    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        if is_softmax(w) or is_partials(w):
            run_softmax(args, w, rank, world, local_rank)
        else:
            run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
