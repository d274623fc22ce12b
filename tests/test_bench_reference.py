"""bench.py --impl reference on CPU: the float64 oracle timed on the host cores prints one
JSON line with our arm's metric, unit, direction and config, a cpu_baseline describing the
run and an e2e object with no host-device bytes."""
import json
import os
import subprocess
import sys

import bench
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    run = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert run.returncode == 0, run.stderr[-2000:]
    lines = [l for l in run.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "suffix tokens/s"
    assert line["higher_is_better"] is True and line["value"] > 0
    cfg = workloads.ATTN_CONFIGS["ragged"]          # our arm's default (headline) workload
    assert line["config"] == bench.attention_config(cfg, workloads.make_layout(cfg), 1)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["steps"] == 1 and line["warmup"] == 1
