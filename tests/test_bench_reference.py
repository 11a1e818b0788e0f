"""The bench's reference arm (CPU): `bench.py --impl reference` times the fp64
oracle on bounded samples of the headline workload and prints one JSON line
with the contract's keys; under torchrun only rank 0 runs and prints."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_the_contract_line():
    res = _run()
    assert res.returncode == 0, res.stderr
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, res.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["metric"] and rec["unit"] == "TFLOP/s" and rec["higher_is_better"] is True
    assert rec["value"] > 0 and rec["steps"] == 1 and rec["warmup"] == 3
    assert rec["dtype"] == "f64" and rec["data"] == "synthetic"
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == rec["value"]
    e2e = rec["e2e"]
    assert e2e["value"] == rec["value"] and e2e["unit"] == rec["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert rec["config"]["L"] == 65536 and rec["config"]["H"] == 12 and rec["config"]["D"] == 128


def test_reference_arm_other_ranks_exit_quietly():
    res = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == ""
