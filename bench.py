"""Benchmark: fused log-prob + entropy forward + backward of the chunked LM head.

One step = lmhead_logps_fwd + lmhead_logps_bwd (logp, entropy, lse, then
d_hidden and d_weight for per-token cotangents of logp and entropy) over one
batch of the workload, through the C ABI.  Default workload: the
Qwen3-4B-shaped head (T = 4096 tokens, H = 2560, V = 151,936, chunk 512,
tau = 1) with synthetic seeded inputs.

Prints ONE JSON line (rank 0).  `value` is tokens/s with inputs resident in
HBM; `e2e` is the same metric with the per-step inputs copied from pinned
host memory (double-buffered: the next step's inputs are copied while this
step computes) and the per-token results copied back inside the timed region.
`roofline` reports the dominant kernel's achieved TFLOP/s (algorithmic flops
per launch / mean launch time from CUDA events on the launching stream)
against the measured dense BF16 peak.  `cpu_baseline` times the fp64 oracle
on a bounded sample of the same workload on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  (N > 1: launched by torch.distributed.run, one independent replica per GPU)
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s and TFLOP/s of fused logp+entropy fwd+bwd; % of GB300 BF16 tensor peak"
UNIT = "tokens/s"
# GEMM kernels and their algorithmic flops per step in units of T_v*H*V
GEMM_KERNELS = {"fwd_stats_gemm": 2.0, "bwd_dz_gemm": 2.0, "bwd_grad_gemm": 4.0,
                "bwd_all_gemm": 6.0, "bwd_window_gemm": 6.0}
# the part of those flops that recomputes the forward's logits
RECOMPUTE = {"bwd_dz_gemm": 2.0, "bwd_all_gemm": 2.0, "bwd_window_gemm": 2.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=150)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_4b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--op", choices=["head", "score_logits"], default="head",
                    help="head: the hidden-state head (default); score_logits: the logits-level entry")
    ap.add_argument("--only-device", action="store_true",
                    help="time the device-resident steps only (profiling runs)")
    return ap.parse_args()


def dist_setup(n):
    import torch
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_inputs(name):
    from chunked_lm_head_tcgen05_gb300 import workloads
    w = workloads.WORKLOADS[name]
    return w, workloads.make_inputs(w)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = sorted(float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit())
        mx = max((float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(rows)}


def kernel_source_hash():
    """Hash of the sources that define the tensor-core GEMM kernels."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunked_lm_head_tcgen05_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f in ("tc_gemm.cuh", "ptx.cuh", "kernels.h") or (f.startswith("gemm_") and f.endswith(".cu")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class OracleSample:
    """The fp64 oracle, as it stands, on the first n tokens of the workload:
    full forward + backward (d_hidden rows and every d_weight row)."""

    def __init__(self, name):
        import oracle
        from chunked_lm_head_tcgen05_gb300 import workloads
        self.w, x = workload_inputs(name)
        self.o = oracle.default()
        self.hb = workloads.bf16_bits(x["hidden"])
        self.wb = workloads.bf16_bits(x["weight"])
        self.y = x["targets"].numpy()
        self.m = None if x["loss_mask"] is None else x["loss_mask"].numpy()
        self.gl = x["grad_logp"].double().numpy()
        self.ge = x["grad_entropy"].double().numpy()

    def run(self, n):
        """Returns (scored tokens, seconds) for one pass over n tokens."""
        import numpy as np
        mm = None if self.m is None else self.m[:n]
        t0 = time.perf_counter()
        self.o.forward(self.hb[:n], self.wb, self.y[:n], mm, self.w.temperature)
        self.o.backward(self.hb[:n], self.wb, self.y[:n], mm, self.w.temperature, self.gl[:n],
                        self.ge[:n])
        dt = time.perf_counter() - t0
        return (n if mm is None else int(np.sum(mm != 0))), dt

    def calibrate(self, seconds):
        """Smallest power-of-two sample that takes about `seconds` (at least 1 token)."""
        T = self.w.T
        n = 1
        _, dt = self.run(n)
        while dt < seconds / 2 and n < min(4096, T):
            n = min(2 * n, T)
            _, dt = self.run(n)
        return n

    def describe(self, n, dt):
        return ("first %d tokens of the %s workload: fp64 forward + backward (all %d d_weight "
                "rows), %.2f s per pass" % (n, self.w.name, self.w.V, dt))


def cublas_same_shape(h, w, stream, reps):
    """Plain bf16 GEMMs (torch.matmul, i.e. cuBLAS; bf16 in and out) of the head's three
    contraction shapes with the [T, V] logits materialised: logits = h W^T,
    d_hidden = dz W, d_weight = dz^T h.  Context for the fused kernels, which never
    hold [T, V] and add their epilogues; not a path of the head."""
    import torch
    T, H = h.shape
    V = w.shape[0]
    gen = torch.Generator(device=h.device).manual_seed(7)
    dz = torch.randn((T, V), device=h.device, dtype=torch.bfloat16, generator=gen)
    z = torch.empty((T, V), device=h.device, dtype=torch.bfloat16)
    dh = torch.empty((T, H), device=h.device, dtype=torch.bfloat16)
    dw = torch.empty((V, H), device=h.device, dtype=torch.bfloat16)
    ops = {"logits": lambda: torch.matmul(h, w.t(), out=z),
           "d_hidden": lambda: torch.matmul(dz, w, out=dh),
           "d_weight": lambda: torch.matmul(dz.t(), h, out=dw)}
    flops = 2.0 * T * H * V
    res = {}
    for name, fn in ops.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        res[name] = {"ms": ms, "tflops": flops / (ms / 1e3) / 1e12}
    del dz, z, dh, dw
    return res


def cpu_model():
    """Host CPU description (model name, or the architecture where /proc has none)."""
    import platform
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip() + " (" + platform.machine() + ")"
    except OSError:
        pass
    return platform.machine()


def cpu_baseline(name, seconds):
    s = OracleSample(name)
    n = s.calibrate(seconds)
    scored, dt = s.run(n)
    return {"value": scored / dt, "unit": UNIT, "cores": s.o.num_threads(), "kind": "oracle",
            "sample": s.describe(n, dt), "affinity_cores": len(os.sched_getaffinity(0)),
            "cpu": cpu_model()}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one pass over a fixed
    sample, sized so that warm-up + timed steps take about two minutes."""
    if rank != 0:
        return
    s = OracleSample(args.workload)
    n = s.calibrate(max(0.5, 120.0 / (args.steps + args.warmup)))
    for _ in range(args.warmup):
        s.run(n)
    tok, sec = 0, 0.0
    for _ in range(args.steps):
        a, dt = s.run(n)
        tok += a
        sec += dt
    v = tok / sec
    w = s.w
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "%s: T=%d, H=%d, V=%d, chunk=%d, tau=%g"
                   % (w.name, w.T, w.H, w.V, w.chunk_size, w.temperature)},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": s.o.num_threads(), "kind": "oracle",
                         "sample": s.describe(n, sec / args.steps)},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_ours(args, rank, world, local):
    import torch
    import chunked_lm_head_tcgen05_gb300 as lm
    lm.build()
    lm.library()
    w, x = workload_inputs(args.workload)
    dev = torch.device("cuda", local)
    T, H, V = w.T, w.H, w.V
    c, tau = w.chunk_size, w.temperature
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    from chunked_lm_head_tcgen05_gb300 import workloads
    Tv = workloads.scored_count(x)
    logp = torch.empty(T, device=dev)
    ent = torch.empty(T, device=dev)
    lse = torch.empty(T, device=dev)
    dh = torch.empty((T, H), device=dev)
    dw = torch.empty((V, H), device=dev)
    ws = torch.empty(max(lm.lmhead_workspace_size(0, T, H, V, c),
                         lm.lmhead_workspace_size(1, T, H, V, c)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(src, on=None):
        st = stream if on is None else on
        rc = lm.lmhead_logps_fwd(src["hidden"], g["weight"], src["targets"], src["loss_mask"], tau,
                                 c, logp, ent, lse, ws, st)
        rc |= lm.lmhead_logps_bwd(src["hidden"], g["weight"], src["targets"], src["loss_mask"],
                                  tau, c, src["grad_logp"], src["grad_entropy"], lse, ent, dh, dw,
                                  0, ws, st)
        if rc:
            raise lm.LmheadError(rc, "step")

    def timed(fn, k):
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / 1e3

    # ---- device-resident timing
    for _ in range(args.warmup):
        step(g)
    torch.cuda.synchronize()
    assert lm.lmhead_read_device_status(ws, stream) == 0
    clocks = ClockSampler(local)
    clocks.start()
    n0 = lm.lmhead_launch_count()
    t = timed(lambda: step(g), args.steps)
    launches = lm.lmhead_launch_count() - n0
    clk = clocks.stop()
    t = max_over_ranks(t, world)
    ms = t / args.steps * 1e3
    value = Tv * world * args.steps / t

    if args.only_device:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": UNIT, "ms_per_step": ms,
                              "steps": args.steps, "warmup": args.warmup, "only_device": True}))
        return

    # ---- per-kernel durations (CUDA events around each launch, same stream)
    lm.lmhead_profile_enable(1)
    timed(lambda: step(g), max(3, args.steps // 4))
    lm.lmhead_profile_enable(0)
    per = {}
    for i in range(lm.lmhead_profile_count()):
        name, kms = lm.lmhead_profile_record(i)
        a = per.setdefault(name, [0, 0.0])
        a[0] += 1
        a[1] += kms
    total_ms = sum(v[1] for v in per.values())
    n_prof_steps = max(3, args.steps // 4)
    dom = max(GEMM_KERNELS, key=lambda k: per.get(k, [0, 0.0])[1])
    dl, dms = per[dom]
    launches_per_step = dl / n_prof_steps
    flops_per_launch = GEMM_KERNELS[dom] * Tv * H * V / launches_per_step
    achieved = flops_per_launch / (dms / dl / 1e3) / 1e12
    peaks, src = measured_peaks()
    peak = peaks["bf16_tflops_sustained"]
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": recorded_traffic(dom, args.workload),
                "peak_source": "%s bf16_tflops_sustained (of %s)" % ("MEASURED_PEAKS.json", src),
                "flops_per_launch": flops_per_launch, "launches_per_step": launches_per_step,
                "frac_without_recompute": achieved / peak
                * (GEMM_KERNELS[dom] - RECOMPUTE.get(dom, 0.0)) / GEMM_KERNELS[dom]}
    kernels = {k: {"launches_per_step": v[0] / n_prof_steps, "ms_per_step": v[1] / n_prof_steps,
                   "share": v[1] / total_ms} for k, v in sorted(per.items())}

    # ---- end to end: per-step inputs from pinned host memory, results back.
    # Two device staging sets: step i+1's inputs are copied on a copy stream
    # while step i computes (as a training loop would prefetch its next batch);
    # each step's logp / entropy are copied back right after it.  The timed
    # region runs from before the first input copy to after the last result copy.
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()
            if k in ("hidden", "targets", "loss_mask", "grad_logp", "grad_entropy")}
    staged = [{k: (torch.empty_like(v, device=dev) if isinstance(v, torch.Tensor) else None)
               for k, v in host.items()} for _ in range(2)]
    out_logp = torch.empty(T, dtype=torch.float32).pin_memory()
    out_ent = torch.empty(T, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values() if isinstance(v, torch.Tensor))
    d2h = 2 * T * 4
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(i):
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(consumed[i % 2])   # step i-2 is done with this set
            for k, v in host.items():
                if isinstance(v, torch.Tensor):
                    staged[i % 2][k].copy_(v, non_blocking=True)
            copied[i % 2].record(copy_stream)

    def e2e_run(k):
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_stream(stream)
        copy_in(0)
        for i in range(k):
            if i + 1 < k:
                copy_in(i + 1)
            stream.wait_event(copied[i % 2])
            step(staged[i % 2])
            consumed[i % 2].record(stream)
            out_logp.copy_(logp, non_blocking=True)
            out_ent.copy_(ent, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / 1e3

    e2e_run(2)
    ne = max(3, args.steps // 2)
    te = max_over_ranks(e2e_run(ne), world)
    e2e_value = Tv * world * ne / te

    # ---- the single-call path (cotangents known up front), strategy chosen by the library
    keep, _ = lm.lmhead_fwd_bwd_keeps_logits(T, H, V, c)
    ws2 = torch.empty(lm.lmhead_workspace_size(2, T, H, V, c), dtype=torch.uint8, device=dev)

    def fused_step():
        rc = lm.lmhead_logps_fwd_bwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau,
                                     c, g["grad_logp"], g["grad_entropy"], logp, ent, lse, dh, dw,
                                     0, 0, ws2, stream)
        if rc:
            raise lm.LmheadError(rc, "fused step")

    for _ in range(2):
        fused_step()
    tf = max_over_ranks(timed(fused_step, max(3, args.steps // 2)), world)
    single_call = {"strategy": "keep_logits" if keep else "recompute",
                   "value": Tv * world * max(3, args.steps // 2) / tf, "unit": UNIT,
                   "ms_per_step": tf / max(3, args.steps // 2) * 1e3,
                   "tflops_counted": 6.0 * Tv * H * V * world * max(3, args.steps // 2) / tf / 1e12}
    del ws2

    # ---- forward alone, backward alone, and the logp-only backward (no entropy cotangent)
    def fwd_only():
        rc = lm.lmhead_logps_fwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau, c,
                                 logp, ent, lse, ws, stream)
        if rc:
            raise lm.LmheadError(rc, "fwd")

    def bwd_only(grad_entropy=g["grad_entropy"]):
        rc = lm.lmhead_logps_bwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau, c,
                                 g["grad_logp"], grad_entropy, lse, ent, dh, dw, 0, ws, stream)
        if rc:
            raise lm.LmheadError(rc, "bwd")

    nb = max(3, args.steps // 4)
    fwd_only()
    tfw = max_over_ranks(timed(fwd_only, nb), world) / nb
    bwd_only()
    tbw = max_over_ranks(timed(bwd_only, nb), world) / nb
    bwd_only(None)
    tbl = max_over_ranks(timed(lambda: bwd_only(None), nb), world) / nb
    fl = Tv * H * V
    splits, tb_rows, vb_cols = lm.lmhead_plan_info(T, H, V, c)
    merge = per.get("fwd_merge")
    merge_bytes = Tv * (16 * splits + 4 + 12 + (4 if g["loss_mask"] is not None else 0))
    breakdown = {
        "fwd": {"ms": tfw * 1e3, "tflops": 2.0 * fl / tfw / 1e12},
        "bwd": {"ms": tbw * 1e3, "tflops_counted": 4.0 * fl / tbw / 1e12,
                "tflops_executed": 6.0 * fl / tbw / 1e12},
        "bwd_logp_only": {"ms": tbl * 1e3, "tflops_counted": 4.0 * fl / tbl / 1e12,
                          "note": "grad_entropy = NULL"},
        "fwd_merge": {"us": merge[1] / merge[0] * 1e3 if merge else None,
                      "bytes": merge_bytes,
                      "gb_per_s": merge_bytes / (merge[1] / merge[0] / 1e3) / 1e9 if merge else None,
                      "note": "%d vocabulary splits; a few microseconds, launch-latency bound at "
                              "this size" % splits},
        "plan": {"fwd_splits": splits, "bwd_tokens": tb_rows, "bwd_vocab": vb_cols},
    }

    # ---- the same step captured once in a CUDA graph and replayed (launch overhead removed)
    graph_replay = None
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(g, side)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            step(g, torch.cuda.current_stream(dev))   # the capturing stream
        cg.replay()
        torch.cuda.synchronize()
        # graph replays and stream-launched steps alternate, so that both see the
        # same power-capped clock
        tgs, tss = [], []
        for _ in range(3):
            tgs.append(max_over_ranks(timed(cg.replay, nb), world) / nb)
            tss.append(max_over_ranks(timed(lambda: step(g), nb), world) / nb)
        tg, ts = sorted(tgs)[1], sorted(tss)[1]
        graph_replay = {"value": Tv * world / tg, "unit": UNIT, "ms_per_step": tg * 1e3,
                        "stream_ms_per_step_interleaved": ts * 1e3}
        del cg
    except Exception as exc:   # report, do not fail the bench
        graph_replay = {"error": str(exc)[:200]}
    stream = torch.cuda.current_stream(dev)

    # ---- device memory: the library allocates nothing; its workspace is bounded by the chunk
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    step(g)
    torch.cuda.synchronize()
    memory = {"workspace_bytes": ws.numel(),
              "peak_delta_during_step_bytes": torch.cuda.max_memory_allocated(dev) - base,
              "logits_bytes_bf16": 2 * T * V,
              "workspace_over_logits": ws.numel() / (2.0 * T * V)}

    # ---- context: the same contractions as plain cuBLAS GEMMs (logits materialised)
    cublas = None
    if 2 * T * V <= (4 << 30):
        cublas = cublas_same_shape(g["hidden"], g["weight"], stream, nb)
        fk = kernels.get("fwd_stats_gemm")
        cublas["fused_fwd_stats_gemm_tflops"] = (2.0 * Tv * H * V / (fk["ms_per_step"] / 1e3) / 1e12
                                                 if fk else None)
        cublas["fused_dominant_kernel"] = {"kernel": roofline["kernel"],
                                           "tflops_executed": roofline["achieved"]}
        cublas["note"] = ("torch.matmul bf16 in / bf16 out on the head's three shapes, [T, V] "
                          "materialised, timed alone; the fused kernels add their epilogues and "
                          "never hold [T, V]")

    counted = 6.0 * Tv * H * V
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s: T=%d (scored %d), H=%d, V=%d, chunk=%d, tau=%g"
                   % (w.name, T, Tv, H, V, c, w.temperature),
                   "T": T, "H": H, "V": V, "chunk_size": c, "temperature": tau,
                   "l2": "inputs larger than L2 (weight %.0f MB bf16 streamed every step)"
                         % (V * H * 2 / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tflops_counted": counted * world / (t / args.steps) / 1e12,
        "tflops_executed": 8.0 * Tv * H * V * world / (t / args.steps) / 1e12,
        "frac_peak_counted": counted / (t / args.steps) / 1e12 / peak,
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "single_call_fwd_bwd": single_call,
        "roofline": roofline,
        "kernels": kernels,
        "breakdown": breakdown,
        "graph_replay": graph_replay,
        "memory": memory,
        "cublas_same_shape": cublas,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_score_logits(args, rank, world, local):
    """Logits-level scoring of one chunk of logits (fp32 [512, 151936], the chunk of the
    Qwen3-4B-shaped head): forward + backward, HBM-bound.  One JSON line."""
    import torch
    import chunked_lm_head_tcgen05_gb300 as lm
    lm.build()
    lm.library()
    dev = torch.device("cuda", local)
    T, V, tau = 512, 151936, 1.0
    g = torch.Generator().manual_seed(20261202)
    z = torch.randn((T, V), generator=g) * 2.0
    z[torch.rand((T, V), generator=g) < 0.01] = float("-inf")
    z = z.to(dev)
    y = torch.randint(0, V, (T,), generator=g, dtype=torch.int64).to(torch.int32).to(dev)
    gl = torch.randn(T, generator=g).to(dev)
    ge = torch.randn(T, generator=g).to(dev)
    logp, ent, lse = (torch.empty(T, device=dev) for _ in range(3))
    dz = torch.empty_like(z)
    stream = torch.cuda.current_stream(dev)

    def step():
        rc = lm.lmhead_score_logits_fwd(z, y, None, tau, logp, ent, lse, stream)
        rc |= lm.lmhead_score_logits_bwd(z, y, None, tau, gl, ge, lse, ent, dz, stream)
        if rc:
            raise lm.LmheadError(rc, "score_logits")

    for _ in range(args.warmup):
        step()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = lm.lmhead_launch_count()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    lm.lmhead_profile_enable(1)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    lm.lmhead_profile_enable(0)
    per = {}
    for i in range(lm.lmhead_profile_count()):
        name, ms = lm.lmhead_profile_record(i)
        per.setdefault(name, []).append(ms)
    peaks, src = measured_peaks()
    bytes_step = 12.0 * T * V
    bwd_ms = sum(per["score_logits_bwd"]) / len(per["score_logits_bwd"])
    achieved = 8.0 * T * V / (bwd_ms / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "tokens/s of logits-level log-prob + entropy scoring, fwd+bwd",
            "value": T * world * args.steps / t, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "logits chunk [512, 151936] fp32, 1% -inf entries, tau=1",
                       "l2": "inputs larger than L2 (311 MB of logits)"},
            "gb_per_s": bytes_step * args.steps / t / 1e9,
            "gpu_launches": lm.lmhead_launch_count() - n0 - 2 * 3,
            "roofline": {"bound": "hbm", "kernel": "score_logits_bwd", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                         "peak_source": "MEASURED_PEAKS.json hbm_gbs (of %s)" % src},
            "kernels_ms": {k: sum(v) / len(v) for k, v in per.items()},
        }), flush=True)


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.op == "score_logits":
        run_score_logits(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
