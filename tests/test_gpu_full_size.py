"""Parity at the full sizes of the benchmark workloads, in the launch
configuration the benchmark times (same shapes, masks, chunk sizes and
temperatures), on outputs the oracle can compute one by one.

* forward: logp / entropy / lse of sampled scored rows against the oracle;
  unscored rows exactly +0.0;
* backward, dense cotangents: sampled rows of d_hidden against the oracle;
  the column sums of d_weight vanish (sum_v dz_v = 0), and a repeat is
  bitwise identical;
* backward, cotangents nonzero on a sample of tokens only: then d_weight
  depends on those tokens alone, so the whole [V, H] d_weight is compared
  with the oracle's, and every other d_hidden row is exactly zero.
"""
import numpy as np
import pytest
import torch

from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import LIMITS, assert_parity, rel_fro, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

NAMES = ["qwen3_4b", "batched_4k", "packed_long_row", "long_trace"]


@pytest.fixture(scope="module", params=NAMES)
def case(request):
    w = W.WORKLOADS[request.param]
    x = W.make_inputs(w)
    return w, x


def _sample_rows(x, n_scored, n_unscored, seed):
    rng = np.random.default_rng(seed)
    T = x["hidden"].shape[0]
    m = np.ones(T, bool) if x["loss_mask"] is None else x["loss_mask"].numpy() != 0
    scored = np.flatnonzero(m)
    unscored = np.flatnonzero(~m)
    a = rng.choice(scored, size=min(n_scored, scored.size), replace=False)
    b = rng.choice(unscored, size=min(n_unscored, unscored.size), replace=False) if unscored.size else []
    return np.sort(a), np.sort(np.asarray(b, dtype=np.int64))


def test_forward_and_dense_backward(case):
    w, x = case
    g = run_gpu(x)
    assert g["fwd_status"] == 0 and g["bwd_status"] == 0
    rows, masked = _sample_rows(x, 40, 16, 1)
    o = run_oracle(x, rows=rows, want_dweight=False)
    e = assert_parity(g, o, rows=rows, keys=("logp", "entropy", "lse", "d_hidden"))
    for k in ("logp", "entropy", "lse"):
        v = g[k][masked]
        assert np.all(v == 0.0) and not np.any(np.signbit(v))
    assert np.all(g["d_hidden"][masked] == 0.0)
    dw = g["d_weight"]
    colsum = np.linalg.norm(dw.sum(axis=0))
    assert colsum <= 1e-2 * np.linalg.norm(dw), (colsum, np.linalg.norm(dw))
    g2 = run_gpu(x)
    for k in ("logp", "entropy", "lse", "d_hidden", "d_weight"):
        assert np.array_equal(g[k], g2[k]), k
    print(w.name, e)


def test_sparse_cotangent_full_dweight(case):
    w, x = case
    rows, _ = _sample_rows(x, 6, 0, 2)
    xs = dict(x)
    keep = torch.zeros(w.T)
    keep[torch.from_numpy(rows)] = 1.0
    xs["grad_logp"] = x["grad_logp"] * keep
    xs["grad_entropy"] = x["grad_entropy"] * keep
    g = run_gpu(xs)
    o = run_oracle(xs, rows=rows)
    e = {"d_weight": rel_fro(g["d_weight"], o["d_weight"]),
         "d_hidden": rel_fro(g["d_hidden"][rows], o["d_hidden"])}
    assert e["d_weight"] <= LIMITS["d_weight"] and e["d_hidden"] <= LIMITS["d_hidden"], e
    others = np.ones(w.T, bool)
    others[rows] = False
    assert np.all(g["d_hidden"][others] == 0.0)
    print(w.name, e)


@pytest.mark.parametrize("name", ["packed_long_row", "long_trace"])
def test_single_call_keep_logits_full_size(name):
    """The single-call path at full size, with the strategy the cost model picks
    (it keeps the logits at chunk 4096): sampled rows and, with cotangents on a
    token sample, the whole d_weight against the oracle."""
    import chunked_lm_head_tcgen05_gb300 as lm
    from gpu_helpers import run_gpu_fwd_bwd
    w = W.WORKLOADS[name]
    keep, _ = lm.lmhead_fwd_bwd_keeps_logits(w.T, w.H, w.V, w.chunk_size)
    assert keep
    x = W.make_inputs(w)
    rows, _ = _sample_rows(x, 6, 0, 3)
    keepmask = torch.zeros(w.T)
    keepmask[torch.from_numpy(rows)] = 1.0
    x["grad_logp"] = x["grad_logp"] * keepmask
    x["grad_entropy"] = x["grad_entropy"] * keepmask
    g = run_gpu_fwd_bwd(x, 0)
    assert g["status"] == 0
    o = run_oracle(x, rows=rows)
    e = assert_parity(g, o, rows=rows, keys=("logp", "entropy", "lse"))
    e["d_weight"] = rel_fro(g["d_weight"], o["d_weight"])
    e["d_hidden"] = rel_fro(g["d_hidden"][rows], o["d_hidden"])
    assert e["d_weight"] <= LIMITS["d_weight"] and e["d_hidden"] <= LIMITS["d_hidden"], e
    print(name, e)


def test_device_memory_bounded_by_chunk(case):
    """Everything the head adds on the device during a forward + backward (its
    workspace included) stays below one bf16 [T, V] logits tensor, and the
    library itself allocates nothing: the peak over the calls equals the
    allocations made before them."""
    import chunked_lm_head_tcgen05_gb300 as lm
    from gpu_helpers import ensure_built, to_device
    ensure_built()
    w, x = case
    g = to_device(x)
    T, H = g["hidden"].shape
    V = g["weight"].shape[0]
    c, tau = x["chunk_size"], x["temperature"]
    logp, ent, lse = (torch.empty(T, device="cuda") for _ in range(3))
    dh = torch.empty((T, H), device="cuda")
    dw = torch.empty((V, H), device="cuda")
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    ws = torch.empty(max(lm.lmhead_workspace_size(0, T, H, V, c),
                         lm.lmhead_workspace_size(1, T, H, V, c)), dtype=torch.uint8,
                     device="cuda")
    after_ws = torch.cuda.memory_allocated()
    assert lm.lmhead_logps_fwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau, c,
                               logp, ent, lse, ws) == 0
    assert lm.lmhead_logps_bwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau, c,
                               g["grad_logp"], g["grad_entropy"], lse, ent, dh, dw, 0, ws) == 0
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated()
    assert peak == after_ws, (peak, after_ws)
    assert peak - base < 2 * T * V, (peak - base, 2 * T * V)
    assert lm.lmhead_read_device_status(ws) == 0


@pytest.mark.parametrize("strategy", ["two_calls", "keep_logits"])
def test_large_vocabulary_64bit_offsets(strategy):
    """A 262,144-entry vocabulary at H = 4096: W is 2 GiB and d_weight 4 GiB, so
    byte offsets pass 2^32 and element offsets approach 2^30.  Sampled rows
    and, with cotangents on a token sample, the whole d_weight (its last rows
    included) against the oracle, for the two-call path and for the single
    call with kept logits."""
    import chunked_lm_head_tcgen05_gb300 as lm
    from gpu_helpers import run_gpu_fwd_bwd
    w = W.WORKLOADS["tiny"].with_(T=700, H=4096, V=262144, chunk_size=2048, temperature=0.9,
                                  mask="bernoulli", mask_drop=0.25, hidden_dist="rms",
                                  weight_std=0.02, seed=51)
    x = W.make_inputs(w)
    rows, _ = _sample_rows(x, 5, 0, 4)
    keepmask = torch.zeros(w.T)
    keepmask[torch.from_numpy(rows)] = 1.0
    x["grad_logp"] = x["grad_logp"] * keepmask
    x["grad_entropy"] = x["grad_entropy"] * keepmask
    if strategy == "two_calls":
        g = run_gpu(x)
        assert g["fwd_status"] == 0 and g["bwd_status"] == 0
    else:
        g = run_gpu_fwd_bwd(x, lm.LMHEAD_STRATEGY_KEEP_LOGITS)
        assert g["status"] == 0
    o = run_oracle(x, rows=rows)
    e = assert_parity(g, o, rows=rows, keys=("logp", "entropy", "lse"))
    e["d_weight"] = rel_fro(g["d_weight"], o["d_weight"])
    e["d_hidden"] = rel_fro(g["d_hidden"][rows], o["d_hidden"])
    e["d_weight_tail"] = rel_fro(g["d_weight"][-4096:], o["d_weight"][-4096:])
    assert max(e["d_weight"], e["d_weight_tail"]) <= LIMITS["d_weight"], e
    assert e["d_hidden"] <= LIMITS["d_hidden"], e
    print(strategy, e)
