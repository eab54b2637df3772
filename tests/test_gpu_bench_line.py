"""bench.py end to end on the GPU (tiny workload, short regions): one JSON line
with every key of the benchmark contract, consistent values, and the
per-workload entries with the oracle beside each."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_has_the_contract_keys():
    d = _run(["--workload", "tiny", "--steps", "5", "--warmup", "3", "--repeats", "3",
              "--no-workloads", "--cpu-seconds", "0.1"])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "clocks",
              "e2e", "gpu_launches", "roofline", "cpu_baseline"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("tiny:")
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert set(d["e2e"]) == {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9 and "traffic" in r
    assert d["repeats"]["regions"] == 3 and len(d["repeats"]["ms_per_step_all"]) == 3
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0
    assert c["parity_on_sample"]["logp"] <= 2e-3


def test_bench_workloads_key():
    d = _run(["--workload", "tiny", "--steps", "3", "--warmup", "3", "--repeats", "1",
              "--cpu-seconds", "0.1", "--workload-cpu-seconds", "0.1"])
    wl = d["workloads"]
    assert list(wl) == ["tiny", "qwen3_4b", "batched_4k", "packed_long_row", "long_trace"]
    for name, w in wl.items():
        assert w["ms_per_step"] > 0 and w["tokens_per_s"] > 0, name
        assert w["oracle"]["kind"] == "oracle", name
        if name != "tiny":
            assert w["oracle"]["scaled"] is True, name
            p = w["oracle"]["parity_on_sample"]
            assert p["logp"] <= 2e-3 and p["d_hidden"] <= 1e-2, name
