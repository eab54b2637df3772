"""Benchmark: fused log-prob + entropy forward + backward of the chunked LM head.

One step = lmhead_logps_fwd + lmhead_logps_bwd (logp, entropy, lse, then
d_hidden and d_weight for per-token cotangents of logp and entropy) over one
batch of the workload, through the C ABI.  Default workload: the
Qwen3-4B-shaped head (T = 4096 tokens, H = 2560, V = 151,936, chunk 512,
tau = 1) with synthetic seeded inputs.

Prints ONE JSON line (rank 0).
- `value`: tokens/s with inputs resident in HBM, the median over `--repeats`
  timed regions of exactly `--steps` steps each (`repeats` gives every
  region's time and the min-max spread).
- `e2e`: the same metric with the per-step inputs copied from pinned host
  memory (double-buffered: the next step's inputs are copied while this step
  computes) and the per-token results copied back inside the timed region.
  Its regions alternate with the device-resident ones, so both see the same
  power-capped clock.
- `clocks`: SM clock, power and clock-event reasons sampled every 10 ms (NVML
  queries from a background thread) during the timed regions.
- `roofline`: the dominant kernel's achieved TFLOP/s (flops per launch / mean
  launch time from CUDA events on the launching stream) against the measured
  dense BF16 peak; the burst figure unless the timed region lasted >= 1 s.
- `cpu_baseline`: the fp64 oracle on a bounded sample of the same workload on
  the host cores.
- `workloads`: every configuration of the head (tiny, Qwen3-4B-shaped,
  batched 4k, packed long row, long trace) with its own timing, dominant
  kernel, clock record and the oracle timed beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  (N > 1: launched by torch.distributed.run, one independent replica per GPU)
"""
import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s and TFLOP/s of fused logp+entropy fwd+bwd; % of GB300 BF16 tensor peak"
UNIT = "tokens/s"
# GEMM kernels and their executed flops per step in units of T_v*H*V
GEMM_KERNELS = {"fwd_stats_gemm": 2.0, "bwd_dz_gemm": 2.0, "bwd_grad_gemm": 4.0,
                "bwd_all_gemm": 6.0, "bwd_window_gemm": 6.0, "fwd_keep_gemm": 2.0}
# the part of those flops that recomputes the forward's logits (executed, not counted)
RECOMPUTE = {"bwd_dz_gemm": 2.0, "bwd_all_gemm": 2.0, "bwd_window_gemm": 2.0}
# configurations of the head, in the order the `workloads` key lists them
ALL_WORKLOADS = ["tiny", "qwen3_4b", "batched_4k", "packed_long_row", "long_trace"]
# a timed region at least this long is compared with the sustained peak, a shorter one
# with the burst peak
SUSTAINED_REGION_S = 1.0


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed regions of --steps steps each (the median is reported)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_4b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="least duration of the oracle's timed sample on the main workload")
    ap.add_argument("--workload-cpu-seconds", type=float, default=4.0,
                    help="least duration of the oracle's timed sample on each other workload")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-configuration `workloads` key")
    ap.add_argument("--op", choices=["head", "score_logits"], default="head",
                    help="head: the hidden-state head (default); score_logits: the logits-level entry")
    ap.add_argument("--only-device", action="store_true",
                    help="time the device-resident steps only (profiling runs)")
    return ap.parse_args(argv)


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


def workload_label(w, scored):
    """The `config.workload` string both arms print for a workload."""
    return ("%s: T=%d (scored %d), H=%d, V=%d, chunk=%d, tau=%g"
            % (w.name, w.T, scored, w.H, w.V, w.chunk_size, w.temperature))


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def bf16_peak(region_s):
    """(peak TFLOP/s, kind, source) for a kernel or step timed over a region of
    `region_s` seconds: the sustained figure for regions of a second or more,
    the burst figure otherwise."""
    peaks, src = measured_peaks()
    kind = "sustained" if region_s >= SUSTAINED_REGION_S else "burst"
    key = "bf16_tflops_sustained" if kind == "sustained" else "bf16_tflops"
    return float(peaks[key]), kind, "MEASURED_PEAKS.json %s (of %s)" % (key, src)


def median(xs):
    return statistics.median(xs) if xs else None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """SM clock, power draw and clock-event reasons of the GPU under test,
    sampled every `period_s` by a background thread.  Query calls only: NVML
    through ctypes (libnvidia-ml, shipped with the driver), or, where that
    cannot be loaded, `nvidia-smi --query-gpu ... -lms`.  Timed regions are
    bracketed by begin()/end(), so the samples taken under load can be
    summarised per region and over all regions."""

    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device, period_s=0.01):
        self.period = period_s
        self.dev = torch_device
        self.samples = []        # (host time, sm MHz, watts, reason bits)
        self.regions = []        # [t0, t1, label]
        self.source = None
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    # -- NVML
    def _nvml_handle(self):
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return None, None
        h = ctypes.c_void_p()
        import torch
        props = torch.cuda.get_device_properties(self.dev)
        tries = []
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            u = str(uuid)
            tries += [("nvmlDeviceGetHandleByUUID", ("GPU-" + u).encode()),
                      ("nvmlDeviceGetHandleByUUID", u.encode())]
        if hasattr(props, "pci_bus_id"):
            bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                        getattr(props, "pci_device_id", 0))
            tries.append(("nvmlDeviceGetHandleByPciBusId_v2", bus.encode()))
        for fn, arg in tries:
            if getattr(nv, fn)(ctypes.c_char_p(arg), ctypes.byref(h)) == 0:
                return nv, h
        n = ctypes.c_uint()
        if nv.nvmlDeviceGetCount_v2(ctypes.byref(n)) == 0 and n.value == 1:
            if nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) == 0:
                return nv, h
        return None, None

    def _nvml_loop(self, nv, h):
        clk, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        reasons = None
        for fn in ("nvmlDeviceGetCurrentClocksEventReasons",
                   "nvmlDeviceGetCurrentClocksThrottleReasons"):
            try:
                reasons = getattr(nv, fn)
                break
            except AttributeError:
                continue
        while not self._stop.is_set():
            t = time.perf_counter()
            ok = nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0   # NVML_CLOCK_SM
            w = mw.value / 1e3 if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0 else None
            r = rs.value if reasons is not None and reasons(h, ctypes.byref(rs)) == 0 else 0
            if ok:
                self.samples.append((t, float(clk.value), w, r))
            self._stop.wait(self.period)

    # -- nvidia-smi fallback (timestamps from the host clock at each line)
    def _smi_loop(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.sw_power_cap,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown")
        idx = os.environ.get("CUDA_VISIBLE_DEVICES", str(self.dev)).split(",")[0] or "0"
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", idx, "--query-gpu=" + q, "--format=csv,noheader,nounits",
                 "-lms", str(max(10, int(self.period * 1e3)))],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        bits = [0x4, 0x8, 0x20, 0x40]
        for line in self._proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                mhz = float(f[0])
                self.max_mhz = float(f[1])
            except ValueError:
                continue
            try:
                w = float(f[2])
            except ValueError:
                w = None
            r = sum(b for b, v in zip(bits, f[3:7]) if v == "Active")
            self.samples.append((time.perf_counter(), mhz, w, r))

    def start(self):
        nv = h = None
        try:
            nv, h = self._nvml_handle()
        except (OSError, AttributeError):
            nv = None
        if nv is not None:
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.source = "nvml every %g ms" % (self.period * 1e3)
            self._thread = threading.Thread(target=self._nvml_loop, args=(nv, h), daemon=True)
        else:
            self.source = "nvidia-smi -lms %d" % max(10, int(self.period * 1e3))
            self._thread = threading.Thread(target=self._smi_loop, daemon=True)
        self._thread.start()
        return self

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def begin(self, label):
        self.regions.append([time.perf_counter(), None, label])
        return len(self.regions) - 1

    def end(self, i):
        self.regions[i][1] = time.perf_counter()

    def _in(self, regions):
        out = []
        for t, mhz, w, r in list(self.samples):
            if any(a <= t <= b for a, b, _ in regions if b is not None):
                out.append((t, mhz, w, r))
        return out

    def region_mhz(self, i):
        s = self._in([self.regions[i]])
        return median([x[1] for x in s])

    def summary(self, labels=None):
        """Clock record of the samples taken inside the regions whose label is in
        `labels` (all regions when None)."""
        regs = [r for r in self.regions if labels is None or r[2] in labels]
        s = self._in(regs)
        if not s:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples_under_load": 0, "source": self.source}
        mhz = sorted(x[1] for x in s)
        bits = 0
        for x in s:
            bits |= x[3]
        watts = [x[2] for x in s if x[2] is not None]
        return {"sm_mhz": median(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if bits & b),
                "samples_under_load": len(s), "sm_mhz_min": mhz[0], "sm_mhz_max": mhz[-1],
                "power_w_max": max(watts) if watts else None,
                "region_s": sum(b - a for a, b, _ in regs if b is not None),
                "source": self.source}


# ------------------------------------------------------------------ recorded ncu traffic
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


# ------------------------------------------------------------------ the oracle on the host
class OracleSample:
    """The fp64 oracle, as it stands, on the first n scored tokens of the
    workload: full forward + backward (their d_hidden rows and every d_weight
    row).  Unscored tokens cost the oracle nothing, so the sample counts scored
    tokens only."""

    def __init__(self, name, inputs=None):
        import numpy as np
        import oracle
        from chunked_lm_head_tcgen05_gb300 import workloads
        if inputs is None:
            self.w, x = workload_inputs(name)
        else:
            self.w, x = inputs["workload"], inputs
        self.o = oracle.default()
        self.hb = workloads.bf16_bits(x["hidden"])
        self.wb = workloads.bf16_bits(x["weight"])
        self.y = x["targets"].numpy()
        m = None if x["loss_mask"] is None else x["loss_mask"].numpy()
        self.rows = np.arange(self.w.T) if m is None else np.nonzero(m)[0]
        self.gl = x["grad_logp"].double().numpy()
        self.ge = x["grad_entropy"].double().numpy()
        self.scored_all = len(self.rows)
        self.last = None

    def run(self, n):
        """Returns (scored tokens, seconds) for one pass over the first n scored tokens."""
        r = self.rows[:n]
        t0 = time.perf_counter()
        fwd = self.o.forward(self.hb[r], self.wb, self.y[r], None, self.w.temperature)
        dh, _ = self.o.backward(self.hb[r], self.wb, self.y[r], None, self.w.temperature,
                                self.gl[r], self.ge[r])
        dt = time.perf_counter() - t0
        self.last = (r, fwd, dh)
        return len(r), dt

    def calibrate(self, seconds):
        """Doubles the sample from one scored token until one pass takes at least
        `seconds` (or covers every scored token); returns (n, scored, seconds) of
        that last pass, which is the measurement."""
        total = self.scored_all
        n = 1
        scored, dt = self.run(n)
        while dt < seconds and n < total:
            n = min(2 * n, total)
            scored, dt = self.run(n)
        return n, scored, dt

    def describe(self, n, dt):
        what = ("all %d scored tokens" % n if n >= self.scored_all
                else "first %d scored tokens" % n)
        return ("%s of the %s workload: fp64 forward + backward (all %d d_weight rows), "
                "%.2f s per pass" % (what, self.w.name, self.w.V, dt))


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


def cpu_baseline(name, seconds, inputs=None):
    s = OracleSample(name, inputs)
    n, scored, dt = s.calibrate(seconds)
    return {"value": scored / dt, "unit": UNIT, "cores": s.o.num_threads(), "kind": "oracle",
            "sample": s.describe(n, dt), "affinity_cores": len(os.sched_getaffinity(0)),
            "cpu": cpu_model()}, s


def sample_parity(s, gpu):
    """Largest differences between the GPU's results and the oracle's on the
    oracle's sampled rows (logp, entropy, lse absolute; d_hidden relative
    Frobenius), a by-product of the timed oracle pass."""
    import numpy as np
    r, (lp, en, ls), dh = s.last
    out = {"rows": int(len(r))}
    for k, ref in (("logp", lp), ("entropy", en), ("lse", ls)):
        a = gpu[k][r]
        fin = np.isfinite(ref)
        out[k] = float(np.abs(a[fin] - ref[fin]).max()) if fin.any() else 0.0
    g = gpu["d_hidden"][r]
    den = float(np.linalg.norm(dh))
    out["d_hidden"] = float(np.linalg.norm(g - dh) / den) if den > 0 else float(np.abs(g).max())
    return out


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one pass over a fixed
    sample, sized so that warm-up + timed steps take about two minutes."""
    if rank != 0:
        return
    s = OracleSample(args.workload)
    n, _, _ = s.calibrate(max(0.5, 60.0 / (args.steps + args.warmup)))
    for _ in range(args.warmup):
        s.run(n)
    tok, sec = 0, 0.0
    for _ in range(args.steps):
        a, dt = s.run(n)
        tok += a
        sec += dt
    v = tok / sec
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_label(s.w, s.scored_all)},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": s.o.num_threads(), "kind": "oracle",
                         "sample": s.describe(n, sec / args.steps)},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------ the GPU arm
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


class Head:
    """One workload resident on the device, with its outputs and workspace, and
    the calls of the head on it."""

    def __init__(self, lm, x, dev, stream):
        import torch
        from chunked_lm_head_tcgen05_gb300 import workloads
        self.lm, self.x, self.dev, self.stream = lm, x, dev, stream
        self.w = w = x["workload"]
        self.T, self.H, self.V = w.T, w.H, w.V
        self.c, self.tau = w.chunk_size, w.temperature
        self.Tv = workloads.scored_count(x)
        self.g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        T, H, V, c = self.T, self.H, self.V, self.c
        self.logp = torch.empty(T, device=dev)
        self.ent = torch.empty(T, device=dev)
        self.lse = torch.empty(T, device=dev)
        self.dh = torch.empty((T, H), device=dev)
        self.dw = torch.empty((V, H), device=dev)
        self.ws = torch.empty(max(lm.lmhead_workspace_size(0, T, H, V, c),
                                  lm.lmhead_workspace_size(1, T, H, V, c)), dtype=torch.uint8,
                              device=dev)
        self.ws2 = None

    def step(self, src=None, on=None):
        lm, g = self.lm, self.g
        src = g if src is None else src
        st = self.stream if on is None else on
        rc = lm.lmhead_logps_fwd(src["hidden"], g["weight"], src["targets"], src["loss_mask"],
                                 self.tau, self.c, self.logp, self.ent, self.lse, self.ws, st)
        rc |= lm.lmhead_logps_bwd(src["hidden"], g["weight"], src["targets"], src["loss_mask"],
                                  self.tau, self.c, src["grad_logp"], src["grad_entropy"],
                                  self.lse, self.ent, self.dh, self.dw, 0, self.ws, st)
        if rc:
            raise lm.LmheadError(rc, "step")

    def fwd_only(self):
        g = self.g
        rc = self.lm.lmhead_logps_fwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"],
                                      self.tau, self.c, self.logp, self.ent, self.lse, self.ws,
                                      self.stream)
        if rc:
            raise self.lm.LmheadError(rc, "fwd")

    def bwd_only(self, with_entropy=True):
        g = self.g
        rc = self.lm.lmhead_logps_bwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"],
                                      self.tau, self.c, g["grad_logp"],
                                      g["grad_entropy"] if with_entropy else None, self.lse,
                                      self.ent, self.dh, self.dw, 0, self.ws, self.stream)
        if rc:
            raise self.lm.LmheadError(rc, "bwd")

    def fused_step(self):
        import torch
        lm, g = self.lm, self.g
        if self.ws2 is None:
            self.ws2 = torch.empty(lm.lmhead_workspace_size(2, self.T, self.H, self.V, self.c),
                                   dtype=torch.uint8, device=self.dev)
        rc = lm.lmhead_logps_fwd_bwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"],
                                     self.tau, self.c, g["grad_logp"], g["grad_entropy"],
                                     self.logp, self.ent, self.lse, self.dh, self.dw, 0, 0,
                                     self.ws2, self.stream)
        if rc:
            raise lm.LmheadError(rc, "fused step")

    def results(self):
        """The last step's per-token results and d_hidden on the host (float64)."""
        return {"logp": self.logp.cpu().double().numpy(),
                "entropy": self.ent.cpu().double().numpy(),
                "lse": self.lse.cpu().double().numpy(),
                "d_hidden": self.dh.cpu().double().numpy()}

    def free(self):
        for k in ("g", "logp", "ent", "lse", "dh", "dw", "ws", "ws2"):
            setattr(self, k, None)


class Timer:
    """Timed regions on one stream: barrier + synchronize on both sides, CUDA
    events on the stream, max over ranks, each region marked in the clock record."""

    def __init__(self, stream, world, clocks):
        self.stream, self.world, self.clocks = stream, world, clocks

    def __call__(self, fn, k, label):
        import torch
        barrier(self.world)
        torch.cuda.synchronize()
        i = self.clocks.begin(label)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for _ in range(k):
            fn()
        e1.record(self.stream)
        torch.cuda.synchronize()
        self.clocks.end(i)
        barrier(self.world)
        return max_over_ranks(e0.elapsed_time(e1) / 1e3, self.world), i


def kernel_profile(lm, timer, fn, k, label):
    """Per-kernel CUDA-event durations over k calls of fn: {name: [launches, ms]}
    and the region's length in seconds."""
    lm.lmhead_profile_enable(1)
    t, _ = timer(fn, k, label)
    lm.lmhead_profile_enable(0)
    per = {}
    for i in range(lm.lmhead_profile_count()):
        name, kms = lm.lmhead_profile_record(i)
        a = per.setdefault(name, [0, 0.0])
        a[0] += 1
        a[1] += kms
    return per, t


def roofline_of(per, steps, Tv, H, V, region_s, workload):
    """Roofline record of the dominant GEMM kernel in a per-kernel profile."""
    gemms = [k for k in GEMM_KERNELS if k in per]
    if not gemms:
        return None
    dom = max(gemms, key=lambda k: per[k][1])
    dl, dms = per[dom]
    launches_per_step = dl / steps
    flops_per_launch = GEMM_KERNELS[dom] * Tv * H * V / launches_per_step
    counted_per_launch = (GEMM_KERNELS[dom] - RECOMPUTE.get(dom, 0.0)) * Tv * H * V / launches_per_step
    launch_s = dms / dl / 1e3
    achieved = flops_per_launch / launch_s / 1e12
    peak, kind, src = bf16_peak(region_s)
    burst, _, _ = bf16_peak(0.0)
    return {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "frac_of_burst_peak": achieved / burst,
            "traffic": recorded_traffic(dom, workload),
            "peak_kind": kind, "peak_source": src, "timed_region_s": region_s,
            "flops_per_launch": flops_per_launch, "launches_per_step": launches_per_step,
            "ms_per_launch": launch_s * 1e3,
            "achieved_counted": counted_per_launch / launch_s / 1e12,
            "frac_counted": counted_per_launch / launch_s / 1e12 / peak,
            "counted_note": ("frac counts the flops the kernel executes (%g T_v H V per step); "
                             "frac_counted leaves out the recompute of the logits (%g T_v H V "
                             "counted)" % (GEMM_KERNELS[dom],
                                               GEMM_KERNELS[dom] - RECOMPUTE.get(dom, 0.0)))}


def kernel_shares(per, steps):
    total = sum(v[1] for v in per.values()) or 1.0
    return {k: {"launches_per_step": v[0] / steps, "ms_per_step": v[1] / steps,
                "share": v[1] / total} for k, v in sorted(per.items())}


def spread(ts):
    return {"min": min(ts), "max": max(ts),
            "spread_pct": 100.0 * (max(ts) - min(ts)) / median(ts) if ts else None}


def measure_workload(lm, name, args, world, dev, stream, clocks, timer, cpu=True):
    """The `workloads` entry of one configuration: fwd + bwd (two calls), forward
    alone, the single-call path where its cost model keeps the logits, the
    dominant kernel, the clock record and the oracle timed beside it."""
    import torch
    t_gen = time.perf_counter()
    w, x = workload_inputs(name)
    t_gen = time.perf_counter() - t_gen
    hd = Head(lm, x, dev, stream)
    Tv, H, V = hd.Tv, hd.H, hd.V
    for _ in range(3):
        hd.step()
    est, _ = timer(hd.step, 1, name + ":probe")
    # regions of about a second or more, at most --steps steps
    k = int(max(3, min(args.steps, math.ceil(1.0 / max(est, 1e-6)))))
    reps = 3
    ts, mhz = [], []
    for _ in range(reps):
        t, i = timer(hd.step, k, name + ":fwd_bwd")
        ts.append(t / k)
        mhz.append(clocks.region_mhz(i))
    step_s = median(ts)
    res = {"config": workload_label(w, Tv), "steps_per_region": k, "regions": reps,
           "ms_per_step": step_s * 1e3, "ms_per_step_all": [t * 1e3 for t in ts],
           "tokens_per_s": Tv * world / step_s,
           "tflops_counted": 6.0 * Tv * H * V / step_s / 1e12,
           "tflops_executed": 8.0 * Tv * H * V / step_s / 1e12}
    peak, kind, _ = bf16_peak(k * step_s)
    res["frac_peak_counted"] = res["tflops_counted"] / peak
    res["peak_kind"] = kind
    cl = clocks.summary({name + ":fwd_bwd"})
    res["clocks"] = cl
    if cl["sm_mhz"]:
        res["tokens_per_s_per_mhz"] = res["tokens_per_s"] / cl["sm_mhz"]
    # forward alone
    hd.fwd_only()
    tf = []
    for _ in range(reps):
        t, _ = timer(hd.fwd_only, k, name + ":fwd")
        tf.append(t / k)
    f = median(tf)
    res["fwd"] = {"ms": f * 1e3, "tokens_per_s": Tv * world / f,
                  "tflops": 2.0 * Tv * H * V / f / 1e12}
    # dominant kernel of the fwd + bwd step
    nk = max(3, k // 2, min(400, int(math.ceil(SUSTAINED_REGION_S / max(step_s, 1e-6)))))
    per, treg = kernel_profile(lm, timer, hd.step, nk, name + ":profile")
    res["roofline"] = roofline_of(per, nk, Tv, H, V, treg, name)
    res["kernels"] = kernel_shares(per, nk)
    # single call (cotangents up front) where the library keeps the logits
    keep, tb = lm.lmhead_fwd_bwd_keeps_logits(hd.T, H, V, hd.c)
    if keep:
        hd.fused_step()
        tk = []
        for _ in range(reps):
            t, _ = timer(hd.fused_step, k, name + ":single_call")
            tk.append(t / k)
        s = median(tk)
        res["single_call_fwd_bwd"] = {"strategy": "keep_logits", "block_tokens": tb,
                                      "ms_per_step": s * 1e3, "tokens_per_s": Tv * world / s,
                                      "tflops_counted": 6.0 * Tv * H * V / s / 1e12,
                                      "speedup_vs_two_calls": step_s / s}
        hd.step()   # leave the two-call results for the parity check below
    else:
        res["single_call_fwd_bwd"] = {"strategy": "recompute (the two calls above)"}
    # the oracle beside it
    if cpu:
        torch.cuda.synchronize()
        gpu = hd.results()
        full = w.T * w.H * w.V <= (1 << 28)
        secs = 1e9 if full else args.workload_cpu_seconds
        base, s = cpu_baseline(name, secs, x)
        n = len(s.last[0])
        o = {"value": base["value"], "unit": UNIT, "cores": base["cores"], "kind": "oracle",
             "sample": base["sample"], "gpu_over_oracle": res["tokens_per_s"] / base["value"]}
        if n >= Tv:
            o["scaled"] = False
        else:
            o["scaled"] = True
            o["scaled_note"] = ("tokens/s of the sampled pass; the oracle's cost is linear in the "
                                "scored tokens, so the whole workload would take %.0f s"
                                % (Tv / base["value"]))
        o["parity_on_sample"] = sample_parity(s, gpu)
        res["oracle"] = o
    res["input_generation_s"] = t_gen
    hd.free()
    del hd, x
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local):
    import torch
    import chunked_lm_head_tcgen05_gb300 as lm
    lm.build()
    lm.library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(local).start()
    timer = Timer(stream, world, clocks)
    w, x = workload_inputs(args.workload)
    hd = Head(lm, x, dev, stream)
    g = hd.g
    T, H, V, Tv = hd.T, hd.H, hd.V, hd.Tv
    c, tau = hd.c, hd.tau
    K, R = args.steps, max(1, args.repeats)

    for _ in range(args.warmup):
        hd.step()
    torch.cuda.synchronize()
    assert lm.lmhead_read_device_status(hd.ws, stream) == 0

    if args.only_device:
        t, _ = timer(hd.step, K, "device")
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": Tv * world * K / t, "unit": UNIT,
                              "ms_per_step": t / K * 1e3, "steps": K, "warmup": args.warmup,
                              "only_device": True}))
        clocks.stop()
        return

    # ---- end-to-end staging: per-step inputs from pinned host memory, results back.
    # Two device staging sets: step i+1's inputs are copied on a copy stream while
    # step i computes (as a training loop prefetches its next batch); each step's
    # logp / entropy are copied back right after it.  The timed region runs from
    # before the first input copy to after the last result copy.
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

    e2e_i = [0]

    def e2e_begin():
        copy_stream.wait_stream(stream)
        copy_in(0)
        e2e_i[0] = 0

    def e2e_one(k):
        i = e2e_i[0]
        if i + 1 < k:
            copy_in(i + 1)
        stream.wait_event(copied[i % 2])
        hd.step(staged[i % 2])
        consumed[i % 2].record(stream)
        out_logp.copy_(hd.logp, non_blocking=True)
        out_ent.copy_(hd.ent, non_blocking=True)
        e2e_i[0] = i + 1

    def e2e_region(k):
        calls = [0]

        def fn():
            if calls[0] == 0:
                e2e_begin()
            e2e_one(k)
            calls[0] += 1
        return timer(fn, k, "e2e")

    e2e_region(2)   # warm the staging path

    # ---- R timed regions of exactly K steps, device-resident and end-to-end alternating
    n0 = lm.lmhead_launch_count()
    t_first, _ = timer(hd.step, K, "device")
    launches = lm.lmhead_launch_count() - n0
    dev_t, dev_mhz, e2e_t = [t_first], [clocks.region_mhz(len(clocks.regions) - 1)], []
    for r in range(R):
        if r > 0:
            t, i = timer(hd.step, K, "device")
            dev_t.append(t)
            dev_mhz.append(clocks.region_mhz(i))
        te, _ = e2e_region(K)
        e2e_t.append(te)
    t_med = median(dev_t)
    ms = t_med / K * 1e3
    value = Tv * world * K / t_med
    e2e_value = Tv * world * K / median(e2e_t)
    step_peak, step_kind, step_src = bf16_peak(t_med)
    clk = clocks.summary({"device", "e2e"})
    clk_dev = clocks.summary({"device"})

    # ---- per-kernel durations (CUDA events around each launch, same stream), over a
    # region of at least a second: the power-capped steady state, against the sustained peak
    nprof = max(3, K // 4, min(400, int(math.ceil(SUSTAINED_REGION_S / max(t_med / K, 1e-6)))))
    per, treg = kernel_profile(lm, timer, hd.step, nprof, "profile")
    roofline = roofline_of(per, nprof, Tv, H, V, treg, args.workload)
    kernels = kernel_shares(per, nprof)

    # ---- the single-call path (cotangents known up front), strategy chosen by the library
    keep, _ = lm.lmhead_fwd_bwd_keeps_logits(T, H, V, c)
    for _ in range(2):
        hd.fused_step()
    nf = max(3, K // 2)
    tf, _ = timer(hd.fused_step, nf, "single_call")
    single_call = {"strategy": "keep_logits" if keep else "recompute",
                   "value": Tv * world * nf / tf, "unit": UNIT, "ms_per_step": tf / nf * 1e3,
                   "tflops_counted": 6.0 * Tv * H * V * world * nf / tf / 1e12}
    hd.ws2 = None

    # ---- forward alone, backward alone, and the logp-only backward (no entropy cotangent)
    nb = max(3, K // 4)
    hd.fwd_only()
    tfw = timer(hd.fwd_only, nb, "fwd")[0] / nb
    hd.bwd_only()
    tbw = timer(hd.bwd_only, nb, "bwd")[0] / nb
    hd.bwd_only(False)
    tbl = timer(lambda: hd.bwd_only(False), nb, "bwd_logp_only")[0] / nb
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

    # ---- the step as two vocabulary shards run in turn on this GPU and combined (what two
    # GPUs would each run, minus the all-gather of the statistics and the all-reduce of the
    # d_hidden shares)
    vocab_shards = None
    try:
        half = (V // 2 + 255) // 256 * 256
        bounds = [(0, half), (half, V)]
        parts = torch.empty((2, T, 4), device=dev)
        shares = [torch.empty((T, H), device=dev) for _ in bounds]
        ws_sh = torch.empty(max(lm.lmhead_workspace_size(op, T, H, b - a, c)
                                for op in (0, 1) for a, b in bounds), dtype=torch.uint8,
                            device=dev)

        def shard_step():
            rc = 0
            for j, (a, b) in enumerate(bounds):
                rc |= lm.lmhead_logps_fwd_shard(g["hidden"], g["weight"][a:b], g["targets"],
                                                g["loss_mask"], a, V, tau, c, parts[j], ws_sh,
                                                stream)
            rc |= lm.lmhead_combine_shards(parts, g["targets"], g["loss_mask"], V, hd.logp,
                                           hd.ent, hd.lse, stream)
            for j, (a, b) in enumerate(bounds):
                rc |= lm.lmhead_logps_bwd_shard(g["hidden"], g["weight"][a:b], g["targets"],
                                                g["loss_mask"], a, V, tau, c, g["grad_logp"],
                                                g["grad_entropy"], hd.lse, hd.ent, shares[j],
                                                hd.dw[a:b], 0, ws_sh, stream)
            if rc:
                raise lm.LmheadError(rc, "shard step")

        shard_step()
        t_sh, t_un = [], []
        for _ in range(3):   # alternating with the unsharded step, at the same clocks
            t_sh.append(timer(shard_step, nb, "vocab_shards")[0] / nb)
            t_un.append(timer(hd.step, nb, "vocab_shards_ref")[0] / nb)
        tsh, tun = median(t_sh), median(t_un)
        vocab_shards = {"shards": [list(b) for b in bounds], "ms_per_step": tsh * 1e3,
                        "unsharded_ms_per_step_interleaved": tun * 1e3,
                        "tokens_per_s": Tv * world / tsh,
                        "note": "two shards' calls in turn on one GPU plus the combine; the "
                                "all-gather of 16 B/token and the all-reduce of d_hidden that "
                                "two GPUs would add are not included"}
        del parts, shares, ws_sh
    except Exception as exc:   # report, do not fail the bench
        vocab_shards = {"error": str(exc)[:200]}

    # ---- the same step captured once in a CUDA graph and replayed (launch overhead removed)
    graph_replay = None
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            hd.step(on=side)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            hd.step(on=torch.cuda.current_stream(dev))   # the capturing stream
        cg.replay()
        torch.cuda.synchronize()
        # graph replays and stream-launched steps alternate, so that both see the
        # same power-capped clock
        tgs, tss = [], []
        for _ in range(3):
            tgs.append(timer(cg.replay, nb, "graph")[0] / nb)
            tss.append(timer(hd.step, nb, "graph_stream")[0] / nb)
        tg, ts = sorted(tgs)[1], sorted(tss)[1]
        graph_replay = {"value": Tv * world / tg, "unit": UNIT, "ms_per_step": tg * 1e3,
                        "stream_ms_per_step_interleaved": ts * 1e3}
        del cg
    except Exception as exc:   # report, do not fail the bench
        graph_replay = {"error": str(exc)[:200]}

    # ---- device memory: the library allocates nothing; its workspace is bounded by the chunk
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    hd.step()
    torch.cuda.synchronize()
    memory = {"workspace_bytes": hd.ws.numel(),
              "peak_delta_during_step_bytes": torch.cuda.max_memory_allocated(dev) - base,
              "logits_bytes_bf16": 2 * T * V,
              "workspace_over_logits": hd.ws.numel() / (2.0 * T * V)}

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
    step_s = t_med / K
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_label(w, Tv),
                   "T": T, "H": H, "V": V, "chunk_size": c, "temperature": tau,
                   "l2": "inputs larger than L2 (weight %.0f MB bf16 streamed every step)"
                         % (V * H * 2 / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "repeats": dict({"regions": len(dev_t), "steps_per_region": K,
                         "ms_per_step_all": [t / K * 1e3 for t in dev_t],
                         "sm_mhz_per_region": dev_mhz,
                         "e2e_ms_per_step_all": [t / K * 1e3 for t in e2e_t],
                         "note": "value and e2e are medians over regions; device and e2e "
                                 "regions alternate"}, **spread([t / K * 1e3 for t in dev_t])),
        "tflops_counted": counted * world / step_s / 1e12,
        "tflops_executed": 8.0 * Tv * H * V * world / step_s / 1e12,
        "frac_peak_counted": counted / step_s / 1e12 / step_peak,
        "frac_peak_executed": 8.0 * Tv * H * V / step_s / 1e12 / step_peak,
        "frac_peak_counted_of_sustained": counted / step_s / 1e12 / bf16_peak(1e9)[0],
        "step_peak": {"tflops": step_peak, "kind": step_kind, "source": step_src,
                      "timed_region_s": t_med},
        "clocks": clk,
        "clocks_device_regions": clk_dev,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "gpu_launches_note": "launches of this library's kernels in one timed region of %d steps"
                             % K,
        "single_call_fwd_bwd": single_call,
        "roofline": roofline,
        "kernels": kernels,
        "breakdown": breakdown,
        "graph_replay": graph_replay,
        "vocab_shards": vocab_shards,
        "memory": memory,
        "cublas_same_shape": cublas,
    }
    if clk_dev.get("sm_mhz"):
        line["tokens_per_s_per_mhz"] = value / clk_dev["sm_mhz"]
    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    main_gpu = hd.results() if do_cpu else None
    hd.free()
    del hd, g, staged, host
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if do_cpu:
        base, s = cpu_baseline(args.workload, args.cpu_seconds, x)
        base["parity_on_sample"] = sample_parity(s, main_gpu)
        line["cpu_baseline"] = base
    del x

    # ---- every configuration of the head, each with the oracle beside it
    if not args.no_workloads:
        wl = {}
        for name in ALL_WORKLOADS:
            if name == args.workload:
                wl[name] = {"config": line["config"]["workload"], "see": "the main line",
                            "steps_per_region": K, "regions": len(dev_t),
                            "ms_per_step": ms, "tokens_per_s": value,
                            "tflops_counted": line["tflops_counted"],
                            "tflops_executed": line["tflops_executed"],
                            "frac_peak_counted": line["frac_peak_counted"],
                            "peak_kind": step_kind,
                            "tokens_per_s_per_mhz": line.get("tokens_per_s_per_mhz"),
                            "fwd": breakdown["fwd"], "single_call_fwd_bwd": single_call,
                            "roofline": roofline, "clocks": clk_dev,
                            "oracle": line.get("cpu_baseline")}
                continue
            wl[name] = measure_workload(lm, name, args, world, dev, stream, clocks, timer,
                                        cpu=do_cpu)
        line["workloads"] = wl
    clocks.stop()
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
    clocks = ClockSampler(local).start()
    timer = Timer(stream, world, clocks)

    def step():
        rc = lm.lmhead_score_logits_fwd(z, y, None, tau, logp, ent, lse, stream)
        rc |= lm.lmhead_score_logits_bwd(z, y, None, tau, gl, ge, lse, ent, dz, stream)
        if rc:
            raise lm.LmheadError(rc, "score_logits")

    for _ in range(args.warmup):
        step()
    n0 = lm.lmhead_launch_count()
    t, _ = timer(step, args.steps, "device")
    launches = lm.lmhead_launch_count() - n0
    per, _ = kernel_profile(lm, timer, step, 3, "profile")
    clocks.stop()
    peaks, src = measured_peaks()
    bytes_step = 12.0 * T * V
    bl, bms = per["score_logits_bwd"]
    achieved = 8.0 * T * V / (bms / bl / 1e3) / 1e9
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
            "gpu_launches": launches,
            "clocks": clocks.summary({"device"}),
            "roofline": {"bound": "hbm", "kernel": "score_logits_bwd", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                         "peak_source": "MEASURED_PEAKS.json hbm_gbs (of %s)" % src},
            "kernels_ms": {k: v[1] / v[0] for k, v in per.items()},
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
