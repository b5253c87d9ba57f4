"""The benchmark's reference arm (the fp64 oracle, timed on the host cores)
runs without a GPU: its JSON line carries the keys the benchmark contract
asks for, and ranks other than 0 exit cleanly without printing."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches")


def _run(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "0"], capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)


def test_reference_line_has_the_contract_keys():
    r = _run(0, 1)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in KEYS:
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith("long")


def test_reference_other_ranks_are_silent():
    r = _run(1, 2)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
