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


def _chunked_loss(lmhead_logps, h, wt, x, w, bounds, **kw):
    y, m = x["targets"].cuda(), x["loss_mask"].cuda()
    gl, ge = x["grad_logp"].cuda(), x["grad_entropy"].cuda()
    loss = 0.0
    for a, b in zip(bounds[:-1], bounds[1:]):
        logp, ent = lmhead_logps(h[a:b], wt, y[a:b].contiguous(), m[a:b].contiguous(),
                                 w.temperature, w.chunk_size, **kw)
        loss = loss + (gl[a:b] * logp).sum() + (ge[a:b] * ent).sum()
    return loss


@pytest.mark.parametrize("via_attribute", [False, True])
def test_per_chunk_calls_accumulate_fp32_main_grad(via_attribute):
    """Five uneven sequence chunks add their weight gradients into one fp32
    buffer inside the library (accumulate_dweight = 1), so the sum is never
    rounded to the parameters' bf16.

    Two checks.  Against the fp64 oracle over the whole sequence the error is
    that of the bf16 logit cotangent (about 2^-9 relative per element, ~1.5e-3
    relative Frobenius after summation), held to 2e-3.  Against one library call
    over the whole sequence, whose d_weight is fp32 throughout, the chunked fp32
    sum differs only by fp32 summation order and the rare bf16 rounding of a
    cotangent whose fp32 value moved by an ulp (lse of a chunk is merged over a
    different number of vocabulary splits): far below 1e-4.  A sum formed in
    bf16 would be off by ~1e-3 there."""
    ensure_built()
    import chunked_lm_head_tcgen05_gb300 as lm
    from chunked_lm_head_tcgen05_gb300.autograd import lmhead_logps
    w, x = _case()
    h = x["hidden"].cuda().requires_grad_(True)
    wt = x["weight"].cuda().requires_grad_(True)
    main = torch.zeros(tuple(wt.shape), dtype=torch.float32, device="cuda")
    bounds = [0, 41, 97, 190, 211, w.T]
    if via_attribute:
        wt.main_grad = main
        loss = _chunked_loss(lmhead_logps, h, wt, x, w, bounds)
    else:
        loss = _chunked_loss(lmhead_logps, h, wt, x, w, bounds, main_grad=main)
    loss.backward()
    assert wt.grad is None
    o = run_oracle(x)
    got = main.double().cpu().numpy()
    assert rel_fro(got, o["d_weight"]) <= 2e-3
    assert rel_fro(h.grad.double().cpu().numpy(), o["d_hidden"]) <= LIMITS["d_hidden"]
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    logp, ent, lse = lm.forward(g["hidden"], g["weight"], g["targets"], g["loss_mask"],
                                w.temperature, w.chunk_size)
    _, dw = lm.backward(g["hidden"], g["weight"], g["targets"], g["loss_mask"], w.temperature,
                        w.chunk_size, g["grad_logp"], g["grad_entropy"], lse, ent)
    assert rel_fro(got, dw.double().cpu().numpy()) <= 1e-4


def test_workspace_is_reused_across_calls():
    ensure_built()
    from chunked_lm_head_tcgen05_gb300 import autograd
    from chunked_lm_head_tcgen05_gb300.autograd import lmhead_logps
    w, x = _case()
    h = x["hidden"].cuda().requires_grad_(True)
    wt = x["weight"].cuda().requires_grad_(True)
    main = torch.zeros(tuple(wt.shape), dtype=torch.float32, device="cuda")
    autograd.release_workspaces()
    _chunked_loss(lmhead_logps, h, wt, x, w, [0, 150, w.T], main_grad=main).backward()
    bufs = {k: v.data_ptr() for k, v in autograd._workspaces.items()}
    assert len(bufs) == 1
    _chunked_loss(lmhead_logps, h, wt, x, w, [0, 100, 200, w.T], main_grad=main).backward()
    assert {k: v.data_ptr() for k, v in autograd._workspaces.items()} == bufs
