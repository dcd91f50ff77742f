"""The benchmark's output contract, checked on the CPU through its reference
arm (the oracle on the host cores): one JSON line with the keys the
benchmark contract names, on the tiny layer."""

import json
import os
import subprocess
import sys

from conftest import ROOT


def test_reference_arm_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config",
         "tiny", "--T", "64", "--steps", "2", "--warmup", "1", "--cpu-tokens", "4"],
        capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    r = json.loads(lines[0])
    for key in ["impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"]:
        assert key in r, key
    assert r["impl"] == "reference" and r["steps"] == 2 and r["value"] > 0
    assert r["higher_is_better"] is True and r["scaling"] == "weak"
    assert r["config"]["workload"].startswith("tiny layer, T=64")
    cb = r["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == r["value"]
    e2e = r["e2e"]
    assert e2e["value"] == r["value"] and e2e["h2d_bytes_per_step"] == 0
