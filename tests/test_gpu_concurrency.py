"""Reentrancy: the library may be called from several host threads at once,
each with its own stream and workspace.  Two threads run forward + backward
on different inputs concurrently (the first calls of each kernel, which
configure it, included); each result must equal the same call made alone,
bit for bit."""
import threading

import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import ensure_built, to_device

pytestmark = pytest.mark.gpu


def _call(x, stream, reps=3):
    g = to_device(x)
    stream.wait_stream(torch.cuda.current_stream())   # the input copies come first
    T, H = g["hidden"].shape
    V = g["weight"].shape[0]
    c, tau = x["chunk_size"], x["temperature"]
    with torch.cuda.stream(stream):
        ws = torch.empty(max(lm.lmhead_workspace_size(0, T, H, V, c),
                             lm.lmhead_workspace_size(1, T, H, V, c)), dtype=torch.uint8,
                         device="cuda")
        out = {k: torch.empty(T, device="cuda") for k in ("logp", "entropy", "lse")}
        out["d_hidden"] = torch.empty((T, H), device="cuda")
        out["d_weight"] = torch.empty((V, H), device="cuda")
        for _ in range(reps):
            rc = lm.lmhead_logps_fwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau,
                                     c, out["logp"], out["entropy"], out["lse"], ws, stream)
            rc |= lm.lmhead_logps_bwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"],
                                      tau, c, g["grad_logp"], g["grad_entropy"], out["lse"],
                                      out["entropy"], out["d_hidden"], out["d_weight"], 0, ws,
                                      stream)
            assert rc == 0
    stream.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["status"] = lm.lmhead_read_device_status(ws, stream)
    return res


def test_two_threads_two_streams():
    ensure_built()
    xs = [W.make_inputs(W.WORKLOADS["tiny"].with_(T=900, H=256, V=3000, chunk_size=64,
                                                  temperature=0.8, mask=m, mask_drop=0.3,
                                                  hidden_dist="rms", weight_std=0.05, seed=s))
          for m, s in (("none", 41), ("bernoulli", 42))]
    results = [None, None]
    errors = []

    def work(i):
        try:
            results[i] = _call(xs[i], torch.cuda.Stream())
        except Exception as e:   # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        alone = _call(xs[i], torch.cuda.Stream(), reps=1)
        assert results[i]["status"] == 0 and alone["status"] == 0
        for k in ("logp", "entropy", "lse", "d_hidden", "d_weight"):
            assert np.array_equal(results[i][k], alone[k], equal_nan=True), (i, k)
