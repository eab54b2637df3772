"""The autograd wrapper: gradients of a loss over logp and entropy against the
fp64 oracle, and the log-prob-only path when the entropy is unused."""
import numpy as np
import pytest
import torch

from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import LIMITS, ensure_built, rel_fro, run_oracle

pytestmark = pytest.mark.gpu


def _case():
    w = W.WORKLOADS["tiny"].with_(T=300, H=192, V=3000, chunk_size=64, temperature=0.7,
                                  mask="bernoulli", mask_drop=0.2, hidden_dist="rms",
                                  weight_std=0.05, seed=44)
    return w, W.make_inputs(w)


@pytest.mark.parametrize("use_entropy", [True, False])
def test_autograd_matches_oracle(use_entropy):
    ensure_built()
    from chunked_lm_head_tcgen05_gb300.autograd import lmhead_logps
    w, x = _case()
    h = x["hidden"].cuda().requires_grad_(True)
    wt = x["weight"].cuda().requires_grad_(True)
    logp, ent = lmhead_logps(h, wt, x["targets"].cuda(), x["loss_mask"].cuda(),
                             w.temperature, w.chunk_size)
    loss = (x["grad_logp"].cuda() * logp).sum()
    if use_entropy:
        loss = loss + (x["grad_entropy"].cuda() * ent).sum()
    loss.backward()
    o = run_oracle(x, grad_entropy=use_entropy)
    assert np.abs(logp.detach().cpu().double().numpy() - o["logp"]).max() <= LIMITS["logp"]
    assert np.abs(ent.detach().cpu().double().numpy() - o["entropy"]).max() <= LIMITS["entropy"]
    # hidden.grad / weight.grad come back in the parameters' dtype (bf16)
    assert rel_fro(h.grad.double().cpu().numpy(), o["d_hidden"]) <= LIMITS["d_hidden"]
    assert rel_fro(wt.grad.double().cpu().numpy(), o["d_weight"]) <= LIMITS["d_weight"]


def test_per_chunk_calls_accumulate_weight_grad():
    """A chunked trainer calls the head once per sequence chunk and sums the
    losses; autograd accumulates the weight's gradient across the calls.  The
    result must match the oracle over the whole sequence."""
    ensure_built()
    from chunked_lm_head_tcgen05_gb300.autograd import lmhead_logps
    w, x = _case()
    h = x["hidden"].cuda().requires_grad_(True)
    wt = x["weight"].cuda().requires_grad_(True)
    y, m = x["targets"].cuda(), x["loss_mask"].cuda()
    gl, ge = x["grad_logp"].cuda(), x["grad_entropy"].cuda()
    bounds = [0, 97, 211, w.T]   # uneven sequence chunks
    loss = 0.0
    for a, b in zip(bounds[:-1], bounds[1:]):
        logp, ent = lmhead_logps(h[a:b], wt, y[a:b].contiguous(), m[a:b].contiguous(),
                                 w.temperature, w.chunk_size)
        loss = loss + (gl[a:b] * logp).sum() + (ge[a:b] * ent).sum()
    loss.backward()
    o = run_oracle(x)
    assert rel_fro(h.grad.double().cpu().numpy(), o["d_hidden"]) <= LIMITS["d_hidden"]
    assert rel_fro(wt.grad.double().cpu().numpy(), o["d_weight"]) <= LIMITS["d_weight"]
