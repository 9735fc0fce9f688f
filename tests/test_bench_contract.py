"""bench.py's command-line contract, on CPU.

The reference arm (the oracle on the host cores) prints one JSON line with the
keys the contract names; the GPU arm has no fallback and exits non-zero when
no CUDA device is present.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=300):
    env = dict(os.environ)
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    import time
    t0 = time.perf_counter()
    r = _run(["--impl", "reference", "--config", "tiny", "--steps", "3", "--warmup", "3"])
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is False and d["unit"] == "ms/iter"
    assert d["value"] > 0.0 and d["value"] == d["ms_per_step"]
    assert d["config"]["workload"].startswith("tiny")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "ms/iter", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # every timed step is real work: the steps fit in the process's own run time
    assert d["ms_per_step"] * d["steps"] / 1e3 <= wall
    # the same config object as the GPU arm's (pairs from the oracle's binning)
    sys.path.insert(0, ROOT)
    import bench
    import gen
    import oracle
    wl = gen.make("tiny")
    args = bench.parse_args(["--config", "tiny"])
    pairs = oracle.count_pairs(wl.splats, wl.depths, wl.width, wl.height)
    assert d["config"] == bench.bench_config(wl, args, pairs, 1)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a CUDA device")
def test_gpu_arm_fails_without_a_device():
    r = _run(["--config", "tiny", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-e2e"])
    assert r.returncode != 0
    assert not any(ln.strip().startswith("{") for ln in r.stdout.splitlines())
