"""bench.py's reference arm on the CPU: `--impl reference` times the float64
oracle on the host cores and prints one JSON line with the same metric, unit
and config as the CUDA arm, plus "impl": "reference", a cpu_baseline block
and an e2e block with zero copy bytes.  Under torchrun only rank 0 prints;
other ranks exit 0 without work.  CPU only."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    env.pop("RANK", None)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                           "--warmup", "3", "--ref-batch-rows", "1"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _run()
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference"
    assert out["metric"] == bench.METRIC and out["unit"] == bench.UNIT
    assert out["config"] == bench.CONFIG
    assert out["higher_is_better"] is True
    assert out["steps"] == 2 and out["warmup"] == 3
    assert out["value"] > 0 and out["ms_per_step"] > 0
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == out["value"] and cb["cores"] >= 1
    assert cb["unit"] == out["unit"] and "batch rows" in cb["sample"]
    e2e = out["e2e"]
    assert e2e["value"] == out["value"] and e2e["unit"] == out["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    r = _run({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
