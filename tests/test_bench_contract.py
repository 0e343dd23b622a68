"""bench.py's reference arm (the CPU oracle timed as the reference) runs on
the CPU: its JSON line must carry the contract's keys, on the same metric,
unit and workload as the GPU arm, and under a multi-rank launch only rank 0
may print it."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.strip()]


def test_reference_arm_json_line():
    lines = _run(["--impl", "reference", "--steps", "3", "--warmup", "3", "--workload", "decode_4k"])
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is False and d["steps"] == 3 and d["warmup"] == 3
    assert d["config"]["workload"] == "decode_4k" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("rank", ["1", "2"])
def test_reference_arm_other_ranks_print_nothing(rank):
    env = {"RANK": rank, "LOCAL_RANK": rank, "WORLD_SIZE": "3", "MASTER_ADDR": "127.0.0.1",
           "MASTER_PORT": "29555"}
    assert _run(["--impl", "reference", "--steps", "3", "--warmup", "3", "--gpus", "3"], env) == []
