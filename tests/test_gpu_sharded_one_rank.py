"""The multi-GPU layer (chunked_lm_head_tcgen05_gb300.sharded) on real kernels:
a one-rank NCCL group on one GPU, so every collective is trivial but every
library call, the exchange code and the autograd function run as they would
on each of several GPUs.  Held to the fp64 oracle."""
import socket
from datetime import timedelta

import numpy as np
import pytest
import torch
import torch.distributed as dist

from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import LIMITS, ensure_built, rel_fro, run_oracle

pytestmark = pytest.mark.gpu


def _port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.fixture
def one_rank_group():
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % _port(), rank=0,
                            world_size=1, timeout=timedelta(seconds=120))
    try:
        yield
    finally:
        dist.destroy_process_group()


def _case():
    w = W.WORKLOADS["tiny"].with_(T=300, H=192, V=3001, chunk_size=64, temperature=0.7, seed=71,
                                  mask="bernoulli", mask_drop=0.2, hidden_dist="rms",
                                  weight_std=0.05)
    return w, W.make_inputs(w)


def test_vocab_parallel_autograd_one_rank(one_rank_group):
    ensure_built()
    from chunked_lm_head_tcgen05_gb300 import sharded
    w, x = _case()
    h = x["hidden"].cuda().requires_grad_(True)
    wt = x["weight"].cuda().requires_grad_(True)
    main = torch.zeros((w.V, w.H), dtype=torch.float32, device="cuda")
    v0, rows = sharded.shard_range(w.V, 0, 1)
    logp, ent = sharded.vocab_parallel_logps(h, wt, x["targets"].cuda(), x["loss_mask"].cuda(),
                                             v0, w.V, w.temperature, w.chunk_size,
                                             main_grad=main)
    loss = (x["grad_logp"].cuda() * logp).sum() + (x["grad_entropy"].cuda() * ent).sum()
    loss.backward()
    o = run_oracle(x)
    assert np.abs(logp.detach().cpu().double().numpy() - o["logp"]).max() <= LIMITS["logp"]
    assert np.abs(ent.detach().cpu().double().numpy() - o["entropy"]).max() <= LIMITS["entropy"]
    assert wt.grad is None
    assert rel_fro(main.double().cpu().numpy(), o["d_weight"]) <= LIMITS["d_weight"]
    assert rel_fro(h.grad.double().cpu().numpy(), o["d_hidden"]) <= LIMITS["d_hidden"]


def test_token_parallel_one_rank(one_rank_group):
    ensure_built()
    from chunked_lm_head_tcgen05_gb300 import sharded
    w, x = _case()
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    logp, ent, lse = sharded.token_parallel_forward(g["hidden"], g["weight"], g["targets"],
                                                    g["loss_mask"], w.temperature, w.chunk_size)
    dh, dw = sharded.token_parallel_backward(g["hidden"], g["weight"], g["targets"],
                                             g["loss_mask"], w.temperature, w.chunk_size,
                                             g["grad_logp"], g["grad_entropy"], lse, ent)
    o = run_oracle(x)
    assert np.abs(lse.cpu().double().numpy() - o["lse"]).max() <= LIMITS["lse"]
    assert rel_fro(dh.cpu().double().numpy(), o["d_hidden"]) <= LIMITS["d_hidden"]
    assert rel_fro(dw.cpu().double().numpy(), o["d_weight"]) <= LIMITS["d_weight"]
