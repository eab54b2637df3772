"""The head inside a CUDA graph: forward + backward captured once and replayed.

Every call enqueues its work on the caller's stream with no host
synchronisation, allocation or configuration call after its first use, so
the sequence can be captured.  Replays must give the eager results bit for
bit, and pick up new input values written into the captured buffers."""
import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import assert_parity, ensure_built, run_oracle, to_device

pytestmark = pytest.mark.gpu


def _buffers(g, T, H, V, c):
    ws = torch.empty(max(lm.lmhead_workspace_size(0, T, H, V, c),
                         lm.lmhead_workspace_size(1, T, H, V, c)), dtype=torch.uint8,
                     device="cuda")
    out = {k: torch.empty(T, device="cuda") for k in ("logp", "entropy", "lse")}
    out["d_hidden"] = torch.empty((T, H), device="cuda")
    out["d_weight"] = torch.empty((V, H), device="cuda")
    return ws, out


def _step(g, out, ws, tau, c):
    rc = lm.lmhead_logps_fwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau, c,
                             out["logp"], out["entropy"], out["lse"], ws)
    rc |= lm.lmhead_logps_bwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau, c,
                              g["grad_logp"], g["grad_entropy"], out["lse"], out["entropy"],
                              out["d_hidden"], out["d_weight"], 0, ws)
    assert rc == 0


def _host(out):
    return {k: v.detach().cpu().double().numpy() for k, v in out.items()}


@pytest.mark.parametrize("mask", ["none", "bernoulli"])
def test_captured_step_replays_eager_bits(mask):
    ensure_built()
    w = W.WORKLOADS["tiny"].with_(T=1000, H=256, V=2800, chunk_size=64, temperature=0.8,
                                  mask=mask, mask_drop=0.3, hidden_dist="rms", weight_std=0.05,
                                  seed=21)
    x = W.make_inputs(w)
    g = to_device(x)
    T, H = g["hidden"].shape
    V = g["weight"].shape[0]
    tau, c = x["temperature"], x["chunk_size"]
    ws, out = _buffers(g, T, H, V, c)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(g, out, ws, tau, c)   # first use: one-time configuration happens here
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = _host(out)
    assert lm.lmhead_read_device_status(ws) == 0

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(g, out, ws, tau, c)
    for k in out:
        out[k].fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    replay = _host(out)
    for k in eager:
        assert np.array_equal(eager[k], replay[k], equal_nan=True), k
    assert lm.lmhead_read_device_status(ws) == 0

    # new values in the captured input buffers: the replay computes on them
    x2 = W.make_inputs(w.with_(seed=22))
    for k in ("hidden", "targets", "grad_logp", "grad_entropy"):
        g[k].copy_(x2[k].to("cuda"))
    if g["loss_mask"] is not None:
        g["loss_mask"].copy_(x2["loss_mask"].to("cuda"))
    graph.replay()
    torch.cuda.synchronize()
    got = _host(out)
    got["fwd_status"] = got["bwd_status"] = lm.lmhead_read_device_status(ws)
    x2["weight"] = x["weight"]
    assert_parity(got, run_oracle(x2))
