"""bench.py --impl reference on the host: the float64 oracle timed on a bounded
sample of the workload, one JSON line with the contract's keys. Rank 0 prints;
other ranks exit without work."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra, *args):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                       capture_output=True, text=True, cwd=ROOT, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return [line for line in r.stdout.splitlines() if line.strip()]


def test_reference_line_keys():
    lines = _run({"RANK": "0", "WORLD_SIZE": "1"}, "--steps", "2", "--warmup", "1")
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "TFLOPS" and d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("c2")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("workload", ["c1", "c4"])
def test_reference_other_workloads(workload):
    d = json.loads(_run({"RANK": "0", "WORLD_SIZE": "1"}, "--workload", workload, "--steps", "1",
                        "--warmup", "0")[0])
    assert d["config"]["workload"].startswith(workload) and d["value"] > 0


def test_reference_other_ranks_print_nothing():
    assert _run({"RANK": "1", "WORLD_SIZE": "2"}, "--gpus", "2", "--steps", "1", "--warmup", "0") == []


def test_gpus_flag_starts_the_ranks_itself():
    """--gpus 2 with no torchrun environment starts two ranks; rank 0 prints
    the one line and reports n_gpus = 2."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "c1"],
                       capture_output=True, text=True, cwd=ROOT, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.strip().startswith("{")]
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"


def test_gpus_flag_must_match_world_size():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, cwd=ROOT, env=env, timeout=300)
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr
    assert not r.stdout.strip()


def test_reference_config_matches_our_arm():
    """Both arms' JSON lines carry the same config object."""
    import bench

    d = json.loads(_run({"RANK": "0", "WORLD_SIZE": "1"}, "--steps", "1", "--warmup", "0")[0])
    assert d["config"] == bench.workload_config("c2", 1)
    for key in ("seed", "l2", "parallelism", "per_rank_batch"):
        assert key in d["config"]
