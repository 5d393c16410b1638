"""bench.py's reference arm (the fp64 oracle on host cores) prints one JSON
line with the contract's keys for every workload family, on a few rows so the
CPU suite stays fast (no GPU involved)."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload", [
    "ln_fwd_bwd_bf16_576000x384", "ln_f32_4096x384", "bwd_rms_bf16_576000x384",
    "fwd_amax_bf16_32768x768", "unet_ln_f16_8192x640", "softmax_bf16_576000x384",
    "partials_bf16_576000x384",
])
def test_reference_arm_line(workload):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", workload, "--rows", "48", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "config", "cpu_baseline", "e2e", "dtype"):
        assert k in line, k
    assert line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith(workload)
