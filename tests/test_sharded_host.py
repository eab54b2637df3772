"""The multi-GPU exchange steps of the head (chunked_lm_head_tcgen05_gb300.sharded),
run as two gloo ranks on the CPU.

The per-rank calls are replaced by an fp64 numpy statement of what each
library call computes for its rows or tokens (``NumpyShardOps``, written from
the definitions); the module under test does only the exchanges: the
all-gather of the vocabulary shards' statistics and their combine in rank
order, the all-reduce of d_hidden (vocabulary-parallel) and of d_weight
(token-parallel).  The composed results must equal the fp64 oracle over the
whole vocabulary and every token, to fp64 rounding."""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LOG2E = 1.0 / math.log(2.0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


class NumpyShardOps:
    """fp64 CPU statement of the library's per-rank calls (test double)."""

    @staticmethod
    def _local(targets, v0, Vs, Vt):
        y = targets.numpy().astype(np.int64)
        y = np.where(y < 0, y + Vt, y)
        valid = (y >= 0) & (y < Vt)
        loc = y - v0
        return valid, np.where(valid & (loc >= 0) & (loc < Vs), loc, -1)

    def shard_forward(self, hidden, weight_shard, targets, loss_mask, v0, Vt, tau, chunk):
        h, w = hidden.double().numpy(), weight_shard.double().numpy()
        u = h @ w.T / tau * LOG2E                      # scaled logits, base-2 units
        m = u.max(axis=1)
        e = np.exp2(u - m[:, None])
        s, s1 = e.sum(axis=1), (e * (u - m[:, None])).sum(axis=1)
        _, loc = self._local(targets, v0, w.shape[0], Vt)
        zy = np.where(loc >= 0, u[np.arange(len(loc)), np.maximum(loc, 0)], -np.inf)
        part = np.stack([m, s, s1, zy], axis=1)
        if loss_mask is not None:
            part[loss_mask.numpy() == 0] = 0.0
        return torch.from_numpy(part)

    def combine(self, partials, targets, loss_mask, Vt):
        p = partials.numpy()                           # [n, T, 4]
        M = p[:, :, 0].max(axis=0)
        wgt = np.exp2(p[:, :, 0] - M)
        s = (wgt * p[:, :, 1]).sum(axis=0)
        s1 = (wgt * (p[:, :, 2] + (p[:, :, 0] - M) * p[:, :, 1])).sum(axis=0)
        zy = p[:, :, 3].max(axis=0)
        valid, _ = self._local(targets, 0, Vt, Vt)
        with np.errstate(divide="ignore", invalid="ignore"):   # unscored rows: zeros, reset below
            l2s = np.log2(s)
            ent = (l2s - s1 / s) / LOG2E
        lse = (M + l2s) / LOG2E
        logp = np.where(valid, (zy - M - l2s) / LOG2E, np.nan)
        if loss_mask is not None:
            off = loss_mask.numpy() == 0
            lse[off], logp[off], ent[off] = 0.0, 0.0, 0.0
        return tuple(torch.from_numpy(a) for a in (logp, ent, lse))

    def shard_backward(self, hidden, weight_shard, targets, loss_mask, v0, Vt, tau, chunk,
                       grad_logp, grad_entropy, lse, entropy, d_weight_shard, accumulate):
        h, w = hidden.double().numpy(), weight_shard.double().numpy()
        z = h @ w.T / tau
        L = lse.numpy()[:, None]
        p = np.exp(z - L)
        _, loc = self._local(targets, v0, w.shape[0], Vt)
        onehot = np.zeros_like(z)
        rows = np.nonzero(loc >= 0)[0]
        onehot[rows, loc[rows]] = 1.0
        gl = grad_logp.numpy()[:, None] if grad_logp is not None else 0.0
        dz = gl * (onehot - p)
        if grad_entropy is not None:
            dz = dz - grad_entropy.numpy()[:, None] * p * (z - L + entropy.numpy()[:, None])
        if loss_mask is not None:
            dz[loss_mask.numpy() == 0] = 0.0
        dz = dz / tau
        dw = dz.T @ h
        if accumulate:
            d_weight_shard += torch.from_numpy(dw)
        else:
            d_weight_shard.copy_(torch.from_numpy(dw))
        return torch.from_numpy(dz @ w)

    def forward(self, hidden, weight, targets, loss_mask, tau, chunk):
        V = weight.shape[0]
        part = self.shard_forward(hidden, weight, targets, loss_mask, 0, V, tau, chunk)
        return self.combine(part[None], targets, loss_mask, V)

    def backward(self, hidden, weight, targets, loss_mask, tau, chunk, grad_logp, grad_entropy,
                 lse, entropy, d_weight, accumulate):
        V = weight.shape[0]
        return self.shard_backward(hidden, weight, targets, loss_mask, 0, V, tau, chunk,
                                   grad_logp, grad_entropy, lse, entropy, d_weight, accumulate)


def _inputs():
    from chunked_lm_head_tcgen05_gb300 import workloads as W
    w = W.WORKLOADS["tiny"].with_(T=40, H=64, V=301, temperature=0.7, mask="bernoulli",
                                  mask_drop=0.3, hidden_dist="rms", weight_std=0.08, seed=77)
    x = W.make_inputs(w)
    y = x["targets"].clone()
    y[3] = -1              # wraps to the last id (in the last shard)
    y[5] = -w.V            # wraps to id 0
    x["targets"] = y
    x["loss_mask"][3] = 1
    x["loss_mask"][5] = 1
    return w, x


def _oracle(x, w):
    import oracle
    from chunked_lm_head_tcgen05_gb300 import workloads as W
    hb, wb = W.bf16_bits(x["hidden"]), W.bf16_bits(x["weight"])
    y, m = x["targets"].numpy(), x["loss_mask"].numpy()
    lp, en, ls = oracle.forward(hb, wb, y, m, w.temperature)
    dh, dw = oracle.backward(hb, wb, y, m, w.temperature, x["grad_logp"].double().numpy(),
                             x["grad_entropy"].double().numpy())
    return lp, en, ls, dh, dw


def _rank(rank, world, port, kind):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from chunked_lm_head_tcgen05_gb300 import sharded
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, x = _inputs()
        o_lp, o_en, o_ls, o_dh, o_dw = _oracle(x, w)
        ops = NumpyShardOps()
        h, W_, y, m = x["hidden"], x["weight"], x["targets"], x["loss_mask"]
        gl, ge = x["grad_logp"].double(), x["grad_entropy"].double()
        if kind == "vocab":
            v0, rows = sharded.shard_range(w.V, rank, world)
            logp, ent, lse = sharded.vocab_parallel_forward(
                h, W_[v0:v0 + rows], y, m, v0, w.V, w.temperature, w.chunk_size, ops=ops)
            dh, dws = sharded.vocab_parallel_backward(
                h, W_[v0:v0 + rows], y, m, v0, w.V, w.temperature, w.chunk_size, gl, ge, lse,
                ent, d_weight_shard=torch.zeros((rows, w.H), dtype=torch.float64), ops=ops)
            np.testing.assert_allclose(logp.numpy(), o_lp, rtol=0, atol=1e-10)
            np.testing.assert_allclose(ent.numpy(), o_en, rtol=0, atol=1e-10)
            np.testing.assert_allclose(lse.numpy(), o_ls, rtol=0, atol=1e-10)
            np.testing.assert_allclose(dh.numpy(), o_dh, rtol=0, atol=1e-12)
            np.testing.assert_allclose(dws.numpy(), o_dw[v0:v0 + rows], rtol=0, atol=1e-12)
        else:
            lo, hi = rank * w.T // world, (rank + 1) * w.T // world
            sl = slice(lo, hi)
            logp, ent, lse = sharded.token_parallel_forward(
                h[sl], W_, y[sl], m[sl], w.temperature, w.chunk_size, ops=ops)
            dwt = torch.zeros((w.V, w.H), dtype=torch.float64)
            dh, dw = sharded.token_parallel_backward(
                h[sl], W_, y[sl], m[sl], w.temperature, w.chunk_size, gl[sl], ge[sl], lse, ent,
                d_weight=dwt, ops=ops)
            np.testing.assert_allclose(logp.numpy(), o_lp[sl], rtol=0, atol=1e-10)
            np.testing.assert_allclose(lse.numpy(), o_ls[sl], rtol=0, atol=1e-10)
            np.testing.assert_allclose(dh.numpy(), o_dh[sl], rtol=0, atol=1e-12)
            np.testing.assert_allclose(dw.numpy(), o_dw, rtol=0, atol=1e-12)
            assert dw is dwt
    finally:
        dist.destroy_process_group()


def _rank_autograd(rank, world, port, use_main):
    """The vocabulary-parallel autograd function: a loss over logp and entropy,
    differentiated through the exchanges, against the oracle."""
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from chunked_lm_head_tcgen05_gb300 import sharded
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, x = _inputs()
        _, _, _, o_dh, o_dw = _oracle(x, w)
        v0, rows = sharded.shard_range(w.V, rank, world)
        # fp64 copies of the bf16 values, so the gradients come back unrounded
        h = x["hidden"].double().requires_grad_(True)
        ws = x["weight"][v0:v0 + rows].double().requires_grad_(True)
        main = torch.zeros((rows, w.H), dtype=torch.float64) if use_main else None
        logp, ent = sharded.vocab_parallel_logps(h, ws, x["targets"], x["loss_mask"], v0, w.V,
                                                 w.temperature, w.chunk_size, ops=NumpyShardOps(),
                                                 main_grad=main)
        loss = (x["grad_logp"].double() * logp).sum() + (x["grad_entropy"].double() * ent).sum()
        loss.backward()
        np.testing.assert_allclose(h.grad.numpy(), o_dh, rtol=0, atol=1e-12)
        got = main.numpy() if use_main else ws.grad.numpy()
        if use_main:
            assert ws.grad is None
        # the shard's gradient buffer is fp32, as the library's d_weight is
        np.testing.assert_allclose(got, o_dw[v0:v0 + rows], rtol=1e-6, atol=1e-12)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("use_main", [False, True])
def test_two_gloo_ranks_vocab_parallel_autograd(use_main):
    mp.start_processes(_rank_autograd, args=(2, _free_port(), use_main), nprocs=2, join=True,
                       start_method="spawn")


@pytest.mark.parametrize("kind", ["vocab", "token"])
def test_two_gloo_ranks_compose_to_the_oracle(kind):
    mp.start_processes(_rank, args=(2, _free_port(), kind), nprocs=2, join=True,
                       start_method="spawn")


def test_shard_ranges_tile_the_vocabulary():
    sys.path.insert(0, ROOT)
    from chunked_lm_head_tcgen05_gb300 import sharded
    for V, n in [(151936, 8), (301, 2), (7, 3), (5, 5)]:
        got = [sharded.shard_range(V, r, n) for r in range(n)]
        assert got[0][0] == 0 and sum(r for _, r in got) == V
        for (a, ra), (b, _) in zip(got, got[1:]):
            assert a + ra == b
        assert max(r for _, r in got) - min(r for _, r in got) <= 1
