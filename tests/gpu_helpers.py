"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI binding and the fp64 oracle on the same seeded inputs, and measure the
differences with the tolerances the head is held to."""
import numpy as np
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads
import oracle

# logp / entropy: absolute; lse: absolute; gradients: relative Frobenius
LIMITS = {"logp": 2e-3, "entropy": 2e-3, "lse": 1e-3, "d_hidden": 1e-2, "d_weight": 1e-2}
# A gradient whose exact value is identically zero (a one-entry vocabulary:
# p = 1, so dz = 0) has no relative error; there the largest |value| is held
# to this absolute bound.  The kernels leave fp32 rounding residue there: p is
# 2^d with d = z log2(e) - lse log2(e) rounded in fp32, |d| ~ 1e-7.
ZERO_REF_ATOL = 1e-4

_built = False


def ensure_built():
    global _built
    if not _built:
        lm.build()
        lm.library()
        _built = True


def to_device(x, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def run_gpu(x, chunk=None, tau=None, grad_entropy=True, grad_logp=True, accumulate=False,
            d_weight_init=None, backward=True):
    """Forward (+ backward) on cuda:0.  Returns numpy arrays and the status."""
    ensure_built()
    g = to_device(x)
    T, H = g["hidden"].shape
    V = g["weight"].shape[0]
    chunk = chunk or x["chunk_size"]
    tau = x["temperature"] if tau is None else tau
    ws = torch.empty(max(lm.lmhead_workspace_size(0, T, H, V, chunk),
                         lm.lmhead_workspace_size(1, T, H, V, chunk)), dtype=torch.uint8,
                     device="cuda")
    logp = torch.empty(T, device="cuda")
    ent = torch.empty(T, device="cuda")
    lse = torch.empty(T, device="cuda")
    rc = lm.lmhead_logps_fwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau, chunk,
                             logp, ent, lse, ws)
    assert rc == 0, lm.STATUS_NAMES.get(rc)
    out = {"fwd_status": lm.lmhead_read_device_status(ws)}
    if backward:
        dh = torch.empty((T, H), device="cuda")
        dw = (torch.empty((V, H), device="cuda") if d_weight_init is None
              else d_weight_init.to("cuda").clone())
        rc = lm.lmhead_logps_bwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau, chunk,
                                 g["grad_logp"] if grad_logp else None,
                                 g["grad_entropy"] if grad_entropy else None, lse,
                                 ent, dh, dw, accumulate, ws)
        assert rc == 0, lm.STATUS_NAMES.get(rc)
        out["bwd_status"] = lm.lmhead_read_device_status(ws)
        out["d_hidden"] = dh.cpu().double().numpy()
        out["d_weight"] = dw.cpu().double().numpy()
    torch.cuda.synchronize()
    out["logp"] = logp.cpu().double().numpy()
    out["entropy"] = ent.cpu().double().numpy()
    out["lse"] = lse.cpu().double().numpy()
    return out


def run_oracle(x, tau=None, grad_entropy=True, grad_logp=True, backward=True, rows=None,
               want_dweight=True):
    """The oracle on the same bf16 inputs (optionally on a subset of rows)."""
    tau = x["temperature"] if tau is None else tau
    hb = workloads.bf16_bits(x["hidden"])
    wb = workloads.bf16_bits(x["weight"])
    y = x["targets"].numpy()
    m = None if x["loss_mask"] is None else x["loss_mask"].numpy()
    gl = x["grad_logp"].double().numpy() if grad_logp else None
    ge = x["grad_entropy"].double().numpy() if grad_entropy else None
    if rows is not None:
        hb, y = hb[rows], y[rows]
        m = None if m is None else m[rows]
        gl = None if gl is None else gl[rows]
        ge = None if ge is None else ge[rows]
    o = {}
    o["logp"], o["entropy"], o["lse"] = oracle.forward(hb, wb, y, m, tau)
    if backward:
        o["d_hidden"], o["d_weight"] = oracle.backward(hb, wb, y, m, tau, gl, ge, want_dweight)
    return o


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def errors(gpu, ora, rows=None, keys=("logp", "entropy", "lse", "d_hidden", "d_weight")):
    e = {}
    for k in keys:
        if k not in ora or ora[k] is None or k not in gpu:
            continue
        a = gpu[k] if rows is None or k == "d_weight" else gpu[k][rows]
        b = ora[k]
        if k in ("d_hidden", "d_weight"):
            e[k] = rel_fro(a, b) if np.any(b != 0) else (float(np.abs(a).max()) if a.size else 0.0)
        else:
            fin = np.isfinite(b)
            assert np.array_equal(np.isfinite(a), fin), "non-finite pattern differs for %s" % k
            e[k] = float(np.abs(a[fin] - b[fin]).max()) if fin.any() else 0.0
    return e


def assert_parity(gpu, ora, rows=None, keys=("logp", "entropy", "lse", "d_hidden", "d_weight")):
    e = errors(gpu, ora, rows, keys)
    zero_ref = {k for k in ("d_hidden", "d_weight")
                if k in e and not np.any(np.asarray(ora[k]) != 0)}
    bad = {k: v for k, v in e.items()
           if not v <= (ZERO_REF_ATOL if k in zero_ref else LIMITS[k])}
    assert not bad, "parity failed: %s (all: %s)" % (bad, e)
    return e


def run_gpu_fwd_bwd(x, strategy, chunk=None, tau=None, grad_entropy=True, grad_logp=True,
                    accumulate=False, d_weight_init=None, with_entropy=True):
    """lmhead_logps_fwd_bwd on cuda:0; numpy results and the device status."""
    ensure_built()
    g = to_device(x)
    T, H = g["hidden"].shape
    V = g["weight"].shape[0]
    chunk = chunk or x["chunk_size"]
    tau = x["temperature"] if tau is None else tau
    ws = torch.empty(lm.lmhead_workspace_size(2, T, H, V, chunk), dtype=torch.uint8,
                     device="cuda")
    logp = torch.empty(T, device="cuda")
    ent = torch.empty(T, device="cuda") if with_entropy else None
    lse = torch.empty(T, device="cuda")
    dh = torch.empty((T, H), device="cuda")
    dw = (torch.empty((V, H), device="cuda") if d_weight_init is None
          else d_weight_init.to("cuda").clone())
    rc = lm.lmhead_logps_fwd_bwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau,
                                 chunk, g["grad_logp"] if grad_logp else None,
                                 g["grad_entropy"] if grad_entropy else None, logp, ent, lse, dh,
                                 dw, accumulate, strategy, ws)
    assert rc == 0, lm.STATUS_NAMES.get(rc)
    out = {"status": lm.lmhead_read_device_status(ws)}
    torch.cuda.synchronize()
    out["logp"] = logp.cpu().double().numpy()
    if with_entropy:
        out["entropy"] = ent.cpu().double().numpy()
    out["lse"] = lse.cpu().double().numpy()
    out["d_hidden"] = dh.cpu().double().numpy()
    out["d_weight"] = dw.cpu().double().numpy()
    return out
