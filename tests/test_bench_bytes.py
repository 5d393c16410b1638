"""bench.py's algorithmic byte model (the denominator of every roofline
fraction) against byte counts written out tensor by tensor: each input read
once, each output written once (workspace partials not counted)."""

import bench
import workloads as W


def test_forward_bytes():
    R, H = 576000, 384
    # x, residual in; sum, y out (bf16); mean, rstd (fp32); gamma, beta, bias (bf16); amax
    want = 2 * R * H * 2 + 2 * R * H * 2 + 2 * R * 4 + 3 * H * 2 + 4
    assert want == 1_774_082_308
    assert bench.fwd_bytes(W.BENCH_LN_BF16_576000x384) == want
    R, H = 32768, 768     # the zero-centered fused add + LN + amax workload
    assert bench.fwd_bytes(W.FWD_AMAX_BF16_32768x768) == 4 * R * H * 2 + 2 * R * 4 + 3 * H * 2 + 4
    R, H = 16384, 8192    # RMSNorm: x, residual in; sum, y out; rstd; gamma
    assert bench.fwd_bytes(W.RMS_BF16_16384x8192) == 4 * R * H * 2 + R * 4 + H * 2
    assert bench.fwd_bytes(W.BENCH_RMS_BF16_16384x8192) == 4 * R * H * 2 + R * 4 + H * 2 + 4
    R, H = 4096, 384      # fp32 LN with bias and residual, no amax
    assert bench.fwd_bytes(W.LN_F32_4096x384) == 4 * R * H * 4 + 2 * R * 4 + 3 * H * 4


def test_backward_bytes():
    R, H = 576000, 384
    # dy, x_sum in, dx out (bf16); mean, rstd in; gamma in; dgamma, dbeta out (fp32)
    want = 3 * R * H * 2 + 2 * R * 4 + H * 2 + 2 * H * 4
    assert want == 1_331_715_840
    assert bench.bwd_bytes(W.BWD_BF16_576000x384_LN) == want
    assert bench.bwd_bytes(W.BWD_BF16_576000x384_RMS) == 3 * R * H * 2 + R * 4 + H * 2 + H * 4
    R, H = 16384, 8192
    assert bench.bwd_bytes(W.RMS_BF16_16384x8192) == 3 * R * H * 2 + R * 4 + H * 2 + H * 4
    for h, w in W.UNET_F16.items():
        assert bench.bwd_bytes(w) == 3 * 8192 * h * 2 + 2 * 8192 * 4 + h * 2 + 2 * h * 4


def test_fp8_dbias_step_bytes():
    R, H = 576000, 384
    w = W.BENCH_LN_FP8_DBIAS_BF16_576000x384
    # the forward also writes one E4M3 byte per element and reads the scale
    assert bench.fwd_bytes(w) == 1_774_082_308 + R * H + 4
    # the backward also writes dbias (fp32)
    assert bench.bwd_bytes(w) == 1_331_715_840 + H * 4


def test_partials_bytes():
    R, H = 576000, 384
    w = W.PARTIALS_BF16_576000x384
    # x in, y out (bf16); three 128-column tiles of (sum, sum of squares)
    # fp32 in; mean, rstd out; gamma, beta in; amax out
    want = 2 * R * H * 2 + R * 3 * 2 * 4 + 2 * R * 4 + 2 * H * 2 + 4
    assert bench.partials_bytes(w, 128) == want
    assert bench.partials_bytes(w, 100) == want + R * 2 * 4   # four tiles


def test_softmax_bytes():
    assert bench.softmax_bytes(W.SMX_BF16_576000x384) == 576000 * 384 * 2 * 2
    assert bench.softmax_bytes(W.SMX_BF16_16384x8192) == 16384 * 8192 * 2 * 2


def test_replica_throughput_counts_every_rank():
    # whole-job rows/s: every replica's rows over the slowest rank's step time
    assert bench.replica_throughput(1000, 4, 2.0) == 4 * 1000 / 2e-3


def test_step_bytes_and_rotation():
    l2 = 129_000_000
    # every [rows, hidden] tensor larger than L2: no rotation
    assert bench.rotation_copies(W.BENCH_LN_BF16_576000x384, l2) == 1
    assert bench.rotation_copies(W.BWD_BF16_576000x384_LN, l2) == 1
    assert bench.rotation_copies(W.BENCH_RMS_BF16_16384x8192, l2) == 1
    # smaller ones cycle through enough buffer sets to move 3 L2s per pass
    for w in (W.LN_F32_4096x384, W.FWD_AMAX_BF16_32768x768, *W.UNET_F16.values()):
        n = bench.rotation_copies(w, l2)
        assert n >= 2 and n * bench.step_bytes(w) >= 3 * l2, (w.name, n)
        assert n == 2 or (n - 1) * bench.step_bytes(w) < 3 * l2, (w.name, n)
    # one-direction workloads count only the call they make
    w = W.FWD_AMAX_BF16_32768x768
    assert bench.step_bytes(w) == bench.fwd_bytes(w)
    w = W.BWD_BF16_576000x384_RMS
    assert bench.step_bytes(w) == bench.bwd_bytes(w)
    w = W.LN_F32_4096x384
    assert bench.step_bytes(w) == bench.fwd_bytes(w) + bench.bwd_bytes(w)


def test_every_configuration_has_a_bench_line_and_an_oracle_step():
    names = set(bench.BENCH_WORKLOADS) | set(bench.CONFIG_WORKLOADS)
    for w in (W.LN_F32_4096x384, W.BWD_BF16_576000x384_LN, W.BWD_BF16_576000x384_RMS,
              W.FWD_AMAX_BF16_32768x768, *W.UNET_F16.values(), W.BENCH_RMS_BF16_16384x8192,
              W.BENCH_LN_BF16_576000x384):
        assert w.name in names, w.name
    for w in bench.CONFIG_WORKLOADS.values():
        small = w.with_(rows=4)
        bench.oracle_step(small, W.make_inputs(small, seed=0), 4)
        assert bench.metric_of(w) == bench.CONFIG_METRIC
