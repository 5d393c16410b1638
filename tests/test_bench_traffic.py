"""The committed ncu traffic record that bench.py reports as `roofline.traffic`:
keyed to the current kernel sources, and every entry close to the algorithmic
bytes of its launch (DRAM writes still dirty in L2 when a kernel ends are not
counted, so entries sit somewhat below)."""

import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RECORD = os.path.join(ROOT, "profiles", "ncu_traffic.json")


def _record():
    with open(RECORD) as f:
        return json.load(f)


def test_record_is_keyed_to_the_current_kernel_sources():
    # A kernel edit needs a new capture of the kernels it changed; entries of
    # kernels it did not change may be carried over to the new hash.
    assert _record()["source_hash"] == bench.source_hash()


def test_entries_are_near_the_algorithmic_bytes():
    d = _record()["workloads"]
    assert d, "no traffic entries"
    for workload, kernels in d.items():
        if workload in bench.SOFTMAX_WORKLOADS:
            w = bench.SOFTMAX_WORKLOADS[workload]
            algo = {"ln_softmax_fwd": bench.softmax_bytes(w)}
        elif workload in bench.PARTIALS_WORKLOADS:
            w = bench.PARTIALS_WORKLOADS[workload]
            algo = {"ln_fwd_from_partials": bench.partials_bytes(w, bench.W.PARTIALS_TILE_COLS)}
        else:
            w = bench.BENCH_WORKLOADS[workload]
            algo = {"ln_fwd": bench.fwd_bytes(w), "ln_bwd": bench.bwd_bytes(w)}
        for kernel, traffic in kernels.items():
            # At most 1.05 of the minimum bytes (no wasted re-reads); the
            # lower bound only catches a capture of the wrong launch.
            ratio = traffic / algo[kernel]
            assert 0.6 <= ratio <= 1.05, (workload, kernel, ratio)


def test_changed_sources_read_as_unmeasured(monkeypatch):
    assert bench.ncu_traffic("ln_fwd_bwd_bf16_576000x384", "ln_fwd") is not None
    monkeypatch.setattr(bench, "source_hash", lambda: "0" * 16)
    assert bench.ncu_traffic("ln_fwd_bwd_bf16_576000x384", "ln_fwd") is None


def test_missing_entry_reads_as_unmeasured():
    assert bench.ncu_traffic("ln_fwd_bwd_bf16_576000x384", "no_such_kernel") is None
