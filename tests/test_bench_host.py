"""The host-only parts of bench.py run on a CPU: the oracle's CPU-baseline
leg (the one part of the default bench line that does not touch the GPU)
and the command line's defaults."""
import sys

import bench
import synth


def test_cpu_baseline_leg_reports_both_figures():
    w = synth.WORKLOADS["tiny"]
    keys, cb, queries, hg = bench._inputs(w, 0)
    cpu = bench.cpu_baseline(w, keys, cb, queries, hg, rows=512, reps=1)
    assert cpu["kind"] == "oracle" and cpu["unit"] == "keys/s" and cpu["value"] > 0
    assert cpu["cores"] >= 1 and cpu["sample"]
    one = cpu["single_thread"]
    assert one["cores"] == 1 and one["value"] > 0


def test_default_command_line(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench._args()
    assert a.gpus == 1 and a.impl == "ours" and a.path == "step"
    assert a.warmup >= 3 and a.workload == bench.DEFAULT_WORKLOAD
