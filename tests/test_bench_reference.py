"""The bench's reference arm (the CPU oracle, timed on a bounded sample)
prints the line the contract asks for: one JSON line with impl "reference",
the same metric, unit, direction and config as the GPU arm would print for
that workload, a cpu_baseline describing the run and an e2e object with no
host-device bytes.  Runs on the CPU, on the oracle-sized workload."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload", ["tiny", "fp8_small"])
def test_reference_arm_line(workload):
    out = subprocess.run(
        [sys.executable, "bench.py", "--impl", "reference", "--workload", workload, "--steps",
         "2", "--warmup", "3"],
        cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    import synth

    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0
    # the same config dict the GPU arm builds from the recipe alone
    assert d["config"] == bench.workload_config(synth.workload(workload), 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
