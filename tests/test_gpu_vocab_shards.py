"""The vocabulary-sharded calls on one GPU: the shards of the table run one
after another, their statistics are combined by lmhead_combine_shards, and the
shard backwards' d_hidden shares are summed (what an all-reduce does across
GPUs).  Held to the fp64 oracle over the whole vocabulary, and to the unsharded
calls on the same inputs."""
import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import LIMITS, assert_parity, ensure_built, rel_fro, run_gpu, run_oracle, \
    to_device

pytestmark = pytest.mark.gpu


def run_sharded(x, bounds, chunk=None, grad_entropy=True):
    """Forward and backward over the shards [bounds[i], bounds[i+1]); numpy results
    and each shard call's device status."""
    ensure_built()
    g = to_device(x)
    T, H = g["hidden"].shape
    V = g["weight"].shape[0]
    chunk = chunk or x["chunk_size"]
    tau = x["temperature"]
    shards = list(zip(bounds[:-1], bounds[1:]))
    parts = torch.full((len(shards), T, 4), float("nan"), device="cuda")
    status = []
    for j, (a, b) in enumerate(shards):
        ws = torch.empty(lm.lmhead_workspace_size(0, T, H, b - a, chunk), dtype=torch.uint8,
                         device="cuda")
        rc = lm.lmhead_logps_fwd_shard(g["hidden"], g["weight"][a:b], g["targets"],
                                       g["loss_mask"], a, V, tau, chunk, parts[j], ws)
        assert rc == 0, lm.STATUS_NAMES.get(rc)
        status.append(lm.lmhead_read_device_status(ws))
    logp, ent, lse = (torch.full((T,), float("nan"), device="cuda") for _ in range(3))
    rc = lm.lmhead_combine_shards(parts, g["targets"], g["loss_mask"], V, logp, ent, lse)
    assert rc == 0, lm.STATUS_NAMES.get(rc)
    dh = torch.zeros((T, H), device="cuda")
    dw = torch.full((V, H), float("nan"), device="cuda")
    for a, b in shards:
        ws = torch.empty(lm.lmhead_workspace_size(1, T, H, b - a, chunk), dtype=torch.uint8,
                         device="cuda")
        share = torch.full((T, H), float("nan"), device="cuda")
        rc = lm.lmhead_logps_bwd_shard(g["hidden"], g["weight"][a:b], g["targets"],
                                       g["loss_mask"], a, V, tau, chunk, g["grad_logp"],
                                       g["grad_entropy"] if grad_entropy else None, lse, ent,
                                       share, dw[a:b], 0, ws)
        assert rc == 0, lm.STATUS_NAMES.get(rc)
        status.append(lm.lmhead_read_device_status(ws))
        dh += share
    torch.cuda.synchronize()
    out = {k: v.cpu().double().numpy() for k, v in
           (("logp", logp), ("entropy", ent), ("lse", lse), ("d_hidden", dh), ("d_weight", dw))}
    out["partials"] = parts.cpu().numpy()
    out["status"] = status
    return out


CASES = {
    "three_ragged_shards_masked": (
        W.WORKLOADS["tiny"].with_(T=300, H=192, V=3001, chunk_size=64, temperature=0.7, seed=61,
                                  mask="bernoulli", mask_drop=0.2, hidden_dist="rms",
                                  weight_std=0.05),
        [0, 1000, 2537, 3001]),
    "two_shards_dense": (
        W.WORKLOADS["tiny"].with_(T=513, H=128, V=2048, chunk_size=16, seed=62,
                                  hidden_dist="rms", weight_std=0.05),
        [0, 1024, 2048]),
    "one_row_shard": (
        W.WORKLOADS["tiny"].with_(T=130, H=64, V=700, chunk_size=8, seed=63, hidden_dist="rms",
                                  weight_std=0.1, mask="bernoulli", mask_drop=0.5),
        [0, 1, 699, 700]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_shards_combine_to_the_whole_vocabulary(name):
    w, bounds = CASES[name]
    x = W.make_inputs(w)
    y = x["targets"].clone()
    y[0], y[1] = -1, -w.V          # wrap to the last id and to id 0
    x["targets"] = y
    if x["loss_mask"] is not None:
        x["loss_mask"][:2] = 1
    got = run_sharded(x, bounds)
    assert got["status"] == [0] * (2 * (len(bounds) - 1))
    assert_parity(got, run_oracle(x))
    # against the unsharded calls: the same arithmetic over other vocabulary splits
    ref = run_gpu(x)
    for k in ("logp", "entropy", "lse"):
        assert np.abs(got[k] - ref[k]).max() <= 2e-5, k
    assert rel_fro(got["d_hidden"], ref["d_hidden"]) <= 1e-3
    assert rel_fro(got["d_weight"], ref["d_weight"]) <= 1e-3
    if x["loss_mask"] is not None:
        off = x["loss_mask"].numpy() == 0
        for k in ("logp", "entropy", "lse"):
            assert np.all(got[k][off] == 0.0)
        assert np.all(got["d_hidden"][off] == 0.0)
        assert np.all(got["partials"][:, off, :] == 0.0)


def test_shards_logp_only_backward():
    w, bounds = CASES["three_ragged_shards_masked"]
    x = W.make_inputs(w)
    got = run_sharded(x, bounds, grad_entropy=False)
    assert_parity(got, run_oracle(x, grad_entropy=False))


def test_shard_target_outside_every_shard():
    w, bounds = CASES["two_shards_dense"]
    x = W.make_inputs(w)
    y = x["targets"].clone()
    y[7] = w.V            # outside [-V, V): invalid
    y[9] = -w.V - 1
    x["targets"] = y
    got = run_sharded(x, bounds)
    assert got["status"][:2] == [6, 6]   # LMHEAD_ERR_BAD_TARGET in each shard's forward
    assert np.isnan(got["logp"][7]) and np.isnan(got["logp"][9])
    ok = np.ones(w.T, bool)
    ok[[7, 9]] = False
    o = run_oracle(x)
    assert np.abs(got["logp"][ok] - o["logp"][ok]).max() <= LIMITS["logp"]
    assert np.abs(got["entropy"] - o["entropy"]).max() <= LIMITS["entropy"]
    assert np.abs(got["lse"] - o["lse"]).max() <= LIMITS["lse"]


def test_shards_full_vocabulary_qwen3_4b_size():
    """Two shards of the 151,936-row table at the Qwen3-4B-shaped size (4096
    tokens, H 2560): the combined forward and the summed / concatenated
    gradients agree with the unsharded calls, which the full-size tests hold to
    the oracle."""
    w = W.WORKLOADS["qwen3_4b"]
    x = W.make_inputs(w)
    got = run_sharded(x, [0, 75968, w.V])
    ref = run_gpu(x)
    assert got["status"] == [0, 0, 0, 0]
    for k in ("logp", "entropy", "lse"):
        assert np.abs(got[k] - ref[k]).max() <= 2e-5, k
    assert rel_fro(got["d_hidden"], ref["d_hidden"]) <= 1e-3
    assert rel_fro(got["d_weight"], ref["d_weight"]) <= 1e-3


def _random_layout(i):
    r = np.random.default_rng(20261202 + 5000 + i)
    T = int(r.choice([1, 7, 129, 256, 257, int(r.integers(300, 700))]))
    H = int(64 * r.integers(1, 6))
    V = int(r.integers(2, 4000))
    n = int(min(V, r.integers(1, 6)))
    cuts = sorted(int(c) for c in r.choice(np.arange(1, V), size=n - 1, replace=False)) if n > 1 else []
    bounds = [0] + cuts + [V]
    mask = str(r.choice(["none", "bernoulli", "prompt_prefix"]))
    extra = {"mask_drop": float(r.uniform(0.05, 0.8))} if mask == "bernoulli" else (
        {"rows": 1} if mask == "prompt_prefix" else {})
    w = W.WORKLOADS["tiny"].with_(T=T, H=H, V=V, chunk_size=int(r.choice([1, 16, 64, 512])),
                                  temperature=float(r.choice([0.5, 0.7, 1.0, 2.0])), mask=mask,
                                  hidden_dist="rms", weight_std=float(r.choice([0.02, 0.05, 0.2])),
                                  seed=int(r.integers(1, 1 << 30)), **extra)
    return w, bounds, bool(r.random() > 0.3)


@pytest.mark.parametrize("i", range(8))
def test_random_shard_layouts(i):
    """Seeded random shapes with 1-5 shards at random cut points."""
    w, bounds, with_entropy = _random_layout(i)
    x = W.make_inputs(w)
    got = run_sharded(x, bounds, grad_entropy=with_entropy)
    assert got["status"] == [0] * (2 * (len(bounds) - 1))
    assert_parity(got, run_oracle(x, grad_entropy=with_entropy))
    ref = run_gpu(x, grad_entropy=with_entropy)
    for k in ("logp", "entropy", "lse"):
        # fp32 summation order differs: a few ulps of the value's own magnitude
        fin = np.isfinite(ref[k])
        tol = 2e-5 * np.maximum(1.0, np.abs(ref[k][fin]))
        assert np.all(np.abs(got[k][fin] - ref[k][fin]) <= tol), (k, bounds)
    print(i, dict(T=w.T, H=w.H, V=w.V, chunk=w.chunk_size, tau=w.temperature, mask=w.mask),
          bounds)
