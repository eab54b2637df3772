"""Host-side checks of bench.py (CPU only): the N > 1 rank logic over gloo
with world size 2, and the reference arm's JSON line (the fp64 oracle timed on
the host), alone and under torch.distributed.run with two ranks."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(1.5 + rank, w)
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True,
                           start_method="spawn")
        assert dict(out) == {0: 2.5, 1: 2.5}


def _run(cmd, env=None):
    e = dict(os.environ, OMP_NUM_THREADS="2", **(env or {}))
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=e)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def test_reference_arm_line():
    lines = _run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                  "--steps", "1", "--warmup", "1"])
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    # the same workload string as the GPU arm prints, so the two lines compare
    sys.path.insert(0, ROOT)
    import bench
    from chunked_lm_head_tcgen05_gb300 import workloads
    assert d["config"]["workload"] == bench.workload_label(workloads.WORKLOADS["tiny"], 256)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_under_torchrun_prints_once():
    lines = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                  "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                  str(_free_port()), "bench.py", "--impl", "reference", "--workload", "tiny",
                  "--gpus", "2", "--steps", "1", "--warmup", "1"])
    assert len(lines) == 1 and lines[0]["impl"] == "reference"


def test_clock_record_counts_samples_inside_timed_regions_only():
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    c.samples = [(0.5, 1000.0, 500.0, 0), (1.5, 1500.0, 900.0, 0x4), (2.5, 1800.0, 1000.0, 0),
                 (3.3, 900.0, 100.0, 0x8), (4.0, 2000.0, 50.0, 0x20)]
    c.regions = [[1.0, 3.0, "device"], [3.2, 3.4, "e2e"]]
    d = c.summary({"device"})
    assert d["samples_under_load"] == 2 and d["sm_mhz"] == 1650.0
    assert d["reasons"] == ["sw_power_cap"] and d["power_w_max"] == 1000.0
    both = c.summary()
    assert both["samples_under_load"] == 3 and both["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert c.region_mhz(1) == 900.0


def test_peak_rule_burst_for_short_regions():
    sys.path.insert(0, ROOT)
    import bench
    peaks, _ = bench.measured_peaks()
    p, kind, _ = bench.bf16_peak(0.14)
    assert kind == "burst" and p == peaks["bf16_tflops"]
    p, kind, _ = bench.bf16_peak(2.0)
    assert kind == "sustained" and p == peaks["bf16_tflops_sustained"]
