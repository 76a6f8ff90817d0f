"""The benchmark's reference arm on CPU: the float64 oracle timed on the host cores.

It prints one JSON line carrying the same metric, unit and workload as the device arm,
with the oracle's own rate as the CPU baseline and zero host-device bytes; under a
multi-rank launch only rank 0 runs it and the other ranks exit cleanly without output.
"""
import json
import os
import subprocess
import sys

from tests.conftest import ROOT


def _run(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           *args], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _run({}, "--config", "tiny", "--steps", "2", "--warmup", "1", "--cpu-budget", "0.2")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny" and d["data"] == "synthetic"
    assert d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # the sample is the same for every step, so the mean step time and the rate agree
    tokens = int(d["config"]["sample"].split()[1])
    assert abs(tokens / (d["ms_per_step"] / 1e3) - d["value"]) <= 1e-6 * d["value"]


def test_reference_arm_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"}, "--config", "tiny", "--steps", "1", "--warmup", "0")
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]
