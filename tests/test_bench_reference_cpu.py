"""bench.py's reference arm on the CPU: the oracle timed on host cores, printed
as one JSON line with the keys the benchmark contract fixes (metric, value,
unit, steps, warm-ups, timing direction, the oracle's own cpu_baseline
description and an end-to-end entry with no host-device traffic).  Run on the
small 128-token workload so that the CPU suite stays short."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*extra):
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--config", "c1_tiny",
           "--steps", "1", "--warmup", "1", *extra]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("pass_", ["forward", "backward"])
def test_reference_arm_prints_the_contract_line(pass_):
    j = _run("--pass", pass_)
    assert j["impl"] == "reference"
    assert j["value"] > 0 and j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert j["n_gpus"] == 1 and j["steps"] == 1 and j["warmup"] == 1
    assert j["dtype"] == "f64" and j["data"] == "synthetic"
    assert "c1_tiny" in j["config"]["workload"]
    cpu = j["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["sample"]
    assert cpu["value"] == j["value"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["unit"] == j["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    if pass_ == "backward":
        assert "backward" in j["metric"]
    else:
        assert j["metric"].startswith("MoE-layer tokens/s")
