"""bench.py's reference arm on CPU: the JSON line it prints, and that ranks other
than 0 print nothing.  The reference arm times the fp64 oracle on the host cores,
so it runs here; the GPU arm's line is checked by the GPU runs themselves."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, env=None):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, cwd=ROOT, timeout=240,
                         env={**os.environ, **(env or {})})
    assert res.returncode == 0, res.stderr[-2000:]
    return [ln for ln in res.stdout.splitlines() if ln.strip()]


@pytest.mark.timeout(300)
def test_reference_arm_prints_one_contract_line():
    lines = run_bench("--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "1")
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] >= 3          # at least 3 warm-up steps
    assert d["n_gpus"] == 1 and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"]["workload"] == "decode_mha_f32_b1_h4_d64_ctx512_p16"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert d["gpu_launches"] == 0


@pytest.mark.timeout(300)
def test_reference_arm_other_ranks_print_nothing():
    lines = run_bench("--impl", "reference", "--config", "1", "--steps", "1", "--warmup", "1",
                      env={"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert lines == []


def test_traffic_is_reported_only_for_the_captured_workload():
    """The committed DRAM-traffic records describe the unmodified workloads; a run that
    changes the workload reports traffic null rather than another workload's bytes."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    name = "gqa_decode_bf16_b32_h32x8_d128_ctx1k-32k_p16"
    base = dict(batch=0, window=0, softcap=0.0, sinks=False, ragged=False, split_tokens=0)
    plain = argparse.Namespace(**base)
    assert bench.workload_traffic(plain, "split_bf16_kernel", name) == \
        bench.traffic_record("split_bf16_kernel", name)
    for change in (dict(batch=8), dict(window=4096), dict(softcap=30.0), dict(sinks=True),
                   dict(ragged=True), dict(split_tokens=2048)):
        args = argparse.Namespace(**{**base, **change})
        assert bench.workload_traffic(args, "split_bf16_kernel", name) is None, change
