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
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_under_torchrun_prints_once():
    lines = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                  "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                  str(_free_port()), "bench.py", "--impl", "reference", "--workload", "tiny",
                  "--gpus", "2", "--steps", "1", "--warmup", "1"])
    assert len(lines) == 1 and lines[0]["impl"] == "reference"
