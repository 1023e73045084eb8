"""The benchmark's reference arm (`bench.py --impl reference`) on CPU: it
times the oracle on bounded samples of the headline workload, on all host
cores, and prints one JSON line with the keys the benchmark contract asks
for; under a multi-rank launch only rank 0 does any work."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench_cores():
    import bench

    return bench.host_cores()


def run_bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = run_bench({}, "--steps", "2", "--warmup", "3", "--ref-rows", "8")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "gpt6.7b_p4x8192x4096_n128" and d["config"]["sample_rows"] == 8
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == bench_cores() and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    # the same metric as the GPU arm's line
    import bench
    assert d["metric"] == bench.METRIC


def test_reference_arm_on_a_nonzero_rank_exits_without_output():
    r = run_bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]
