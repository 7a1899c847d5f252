"""The benchmark's JSON contract, checked on CPU through its reference arm.

``bench.py --impl reference`` times the CPU oracle on a bounded sample of the
decode batch and prints one JSON line with the same metric, unit, config and
direction as the GPU arm, plus its own cpu_baseline and e2e objects.  Under a
multi-rank launch only rank 0 runs it; every other rank exits 0 silently.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None, args=()):
    env = dict(os.environ)
    for key in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(key, None)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                          capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)


def test_reference_arm_prints_one_contract_line():
    import bench
    r = _run(args=("--steps", "1", "--warmup", "3"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "rows/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["scaling"] == "weak" and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("decode batch")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e == {"value": d["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_silently():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, ("--steps", "1", "--warmup", "3"))
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_warmup_is_at_least_three():
    r = _run(args=("--steps", "1", "--warmup", "0"))
    assert r.returncode == 0, r.stderr[-2000:]
    assert json.loads(r.stdout.strip().splitlines()[-1])["warmup"] == 3


@pytest.mark.parametrize("flags", [[], ["--sweep"]])
def test_gpu_modes_refuse_without_a_gpu(flags):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *flags], capture_output=True, text=True,
                       cwd=ROOT, timeout=600)
    assert r.returncode != 0 and "no CPU fallback" in (r.stdout + r.stderr)


def test_cpu_baseline_sample_is_bounded_by_time_and_runs():
    import bench
    import workloads
    case = workloads.decode_batch()
    sub = workloads.DecodeCase(case.name, case.logits[:4], case.kv_lens[:4 // case.next_n], case.next_n,
                               case.compress_ratio, case.k)
    secs, cores, runs, total = bench.time_oracle(sub, 1, 3, 0.2)
    assert cores == 1 and secs > 0 and runs >= 3 and total >= 0.2
    secs, cores, runs, total = bench.time_oracle(sub, 1, 2, 1e9, max_runs=4)
    assert runs == 4
