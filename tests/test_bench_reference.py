"""bench.py's reference arm (the fp64 oracle on the host cores) keeps the JSON-line
contract on a CPU-only host: one line with the same metric, unit and direction as the
GPU arm, its workload, a cpu_baseline describing the run and an e2e with no copies; an
unavailable line for a rule with no CPU arm; nothing from ranks other than 0."""
import json
import os
import subprocess
import sys
from pathlib import Path

import bench

ROOT = Path(__file__).resolve().parents[1]


def _run(*args, env=None):
    e = dict(os.environ, **(env or {}))
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", *args], cwd=ROOT,
                       capture_output=True, text=True, env=e, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]


def test_reference_line_contract():
    (line,) = _run("--steps", "3", "--warmup", "3")
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT and line["higher_is_better"] is True
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["steps"] == 3 and line["warmup"] == 3
    assert line["n_gpus"] == 1 and line["vs_baseline"] is None and line["scaling"] == "weak"
    assert line["config"]["workload"] == bench.DEFAULT_WORKLOAD
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_unavailable_and_other_ranks():
    (line,) = _run("--rule", "kv_compact", "--steps", "3", "--warmup", "3")
    assert line["impl"] == "reference" and line["unavailable"]
    assert _run("--steps", "3", "--warmup", "3", env={"RANK": "1", "WORLD_SIZE": "2"}) == []
