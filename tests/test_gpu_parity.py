"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle,
element by element, at sizes the oracle finishes in seconds: several tiles,
ragged tails in T, V and H, masks, temperatures, and the degenerate cases."""
import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import assert_parity, errors, run_gpu, run_oracle, to_device, ensure_built

pytestmark = pytest.mark.gpu

TINY = W.WORKLOADS["tiny"]


def _w(T, H, V, chunk, tau, mask="none", seed=7, **kw):
    return TINY.with_(T=T, H=H, V=V, chunk_size=chunk, temperature=tau, mask=mask, seed=seed, **kw)


def test_tiny_workload():
    """256 tokens, H=128, V=2048, chunk 64: full forward and backward."""
    x = W.make_inputs(TINY)
    g = run_gpu(x)
    o = run_oracle(x)
    e = assert_parity(g, o)
    assert g["fwd_status"] == 0 and g["bwd_status"] == 0
    print("tiny", e)


RAGGED = [
    # T, H, V, chunk, tau, mask, extra
    (333, 192, 3001, 64, 0.7, "bernoulli", dict(mask_drop=0.3)),
    (130, 64, 257, 1000, 1.0, "none", {}),
    (1, 128, 100, 1, 1.0, "none", {}),
    (700, 256, 5000, 128, 0.5, "prompt_prefix", dict(rows=2)),
    (257, 320, 1025, 7, 1.3, "none", {}),
    (520, 128, 2304, 37, 0.9, "packed_pads", dict(pad_tokens=140, segments=5)),
]


@pytest.mark.parametrize("T,H,V,chunk,tau,mask,extra", RAGGED,
                         ids=["T%d_H%d_V%d_c%d" % r[:4] for r in RAGGED])
def test_ragged_shapes(T, H, V, chunk, tau, mask, extra):
    w = _w(T, H, V, chunk, tau, mask, hidden_dist="rms", weight_std=0.05, **extra)
    x = W.make_inputs(w)
    g = run_gpu(x)
    o = run_oracle(x)
    e = assert_parity(g, o)
    print(w, e)


def test_logp_only_and_missing_cotangents():
    """grad_entropy NULL is the log-prob-only backward; grad_logp NULL means zeros."""
    w = _w(300, 128, 1500, 50, 0.7, "bernoulli", mask_drop=0.2, hidden_dist="rms")
    x = W.make_inputs(w)
    g = run_gpu(x, grad_entropy=False)
    assert_parity(g, run_oracle(x, grad_entropy=False))
    g = run_gpu(x, grad_logp=False)
    assert_parity(g, run_oracle(x, grad_logp=False))


def test_unscored_rows_are_exact_zeros_and_never_read():
    w = _w(260, 128, 1000, 32, 0.7, "bernoulli", mask_drop=0.4, hidden_dist="rms")
    x = W.make_inputs(w)
    m = x["loss_mask"].bool()
    g0 = run_gpu(x)
    x_nan = dict(x)
    h = x["hidden"].clone()
    h[~m] = float("nan")
    x_nan["hidden"] = h
    g1 = run_gpu(x_nan)
    mk = ~m.numpy()
    for k in ("logp", "entropy", "lse"):
        assert np.all(g1[k][mk] == 0.0) and not np.any(np.signbit(g1[k][mk]))
        assert np.array_equal(g0[k], g1[k])
    assert np.all(g1["d_hidden"][mk] == 0.0)
    assert np.array_equal(g0["d_weight"], g1["d_weight"])
    assert np.array_equal(g0["d_hidden"], g1["d_hidden"])


def test_negative_targets_wrap_bit_exact():
    w = _w(200, 64, 700, 16, 1.0)
    x = W.make_inputs(w)
    xn = dict(x)
    y = x["targets"].clone()
    y[::3] -= w.V
    xn["targets"] = y
    a, b = run_gpu(x), run_gpu(xn)
    for k in ("logp", "entropy", "lse", "d_hidden", "d_weight"):
        assert np.array_equal(a[k], b[k]), k


def test_invalid_targets():
    """A scored id outside [-V, V): logp NaN, status BAD_TARGET, the rest unchanged."""
    w = _w(150, 64, 600, 16, 1.0)
    x = W.make_inputs(w)
    xb = dict(x)
    y = x["targets"].clone()
    y[5], y[77] = w.V, -w.V - 3
    xb["targets"] = y
    a, b = run_gpu(x), run_gpu(xb)
    assert b["fwd_status"] == 6 and b["bwd_status"] == 6 and a["fwd_status"] == 0
    assert np.isnan(b["logp"][5]) and np.isnan(b["logp"][77])
    keep = np.ones(150, bool)
    keep[[5, 77]] = False
    assert np.array_equal(a["logp"][keep], b["logp"][keep])
    assert np.array_equal(a["entropy"], b["entropy"]) and np.array_equal(a["lse"], b["lse"])
    o = run_oracle(xb)
    assert_parity(b, o)


def test_all_tokens_unscored():
    w = _w(100, 64, 500, 16, 1.0, "all")
    x = W.make_inputs(w)
    g = run_gpu(x, d_weight_init=torch.full((500, 64), 3.0))
    for k in ("logp", "entropy", "lse", "d_hidden", "d_weight"):
        assert np.all(g[k] == 0.0), k
    g = run_gpu(x, accumulate=True, d_weight_init=torch.full((500, 64), 3.0))
    assert np.all(g["d_weight"] == 3.0)


def test_zero_tokens():
    ensure_built()
    V, H = 300, 64
    w = torch.zeros((V, H), dtype=torch.bfloat16, device="cuda")
    h = torch.zeros((0, H), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(0, dtype=torch.int32, device="cuda")
    e = torch.zeros(0, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    assert lm.lmhead_logps_fwd(h, w, y, None, 1.0, 8, e, e, e, ws) == 0
    dw = torch.full((V, H), 5.0, device="cuda")
    dh = torch.zeros((0, H), device="cuda")
    assert lm.lmhead_logps_bwd(h, w, y, None, 1.0, 8, e, e, e, e, dh, dw, 0, ws) == 0
    torch.cuda.synchronize()
    assert torch.all(dw == 0)


def test_deterministic_repeat():
    w = _w(600, 256, 4000, 100, 0.7, "bernoulli", mask_drop=0.1, hidden_dist="rms")
    x = W.make_inputs(w)
    a, b = run_gpu(x), run_gpu(x)
    for k in ("logp", "entropy", "lse", "d_hidden", "d_weight"):
        assert np.array_equal(a[k], b[k]), k


def test_chunk_size_invariance():
    """Chunking changes only the f32 summation order of the gradients
    (tunix PR #2876: 4096 vs 1024 agree within f32 summation order)."""
    w = _w(1100, 128, 9000, 64, 1.0, hidden_dist="rms")
    x = W.make_inputs(w)
    runs = [run_gpu(x, chunk=c) for c in (16, 64, 512, 4096)]
    for r in runs[1:]:
        for k in ("logp", "entropy", "lse"):
            assert np.array_equal(r[k], runs[0][k]), k   # forward does not depend on chunk
        for k in ("d_hidden", "d_weight"):
            d = np.linalg.norm(r[k] - runs[0][k]) / np.linalg.norm(runs[0][k])
            assert d < 1e-3, (k, d)


def test_accumulate_dweight():
    w = _w(300, 128, 1000, 16, 1.0, hidden_dist="rms")
    x = W.make_inputs(w)
    base = run_gpu(x)
    acc = run_gpu(x, accumulate=True, d_weight_init=torch.from_numpy(base["d_weight"]).float())
    d = np.linalg.norm(acc["d_weight"] - 2 * base["d_weight"]) / np.linalg.norm(base["d_weight"])
    assert d < 1e-5


def test_instrumentation_counts_and_names():
    ensure_built()
    w = _w(256, 128, 2048, 64, 1.0)
    x = W.make_inputs(w)
    n0 = lm.lmhead_launch_count()
    lm.lmhead_profile_enable(1)
    run_gpu(x)
    lm.lmhead_profile_enable(0)
    n = lm.lmhead_profile_count()
    names = [lm.lmhead_profile_record(i)[0] for i in range(n)]
    assert lm.lmhead_launch_count() - n0 == n
    for k in ("fwd_stats_gemm", "fwd_merge", "bwd_prep"):
        assert k in names
    # the backward GEMMs: one persistent launch, or two launches per block
    assert "bwd_all_gemm" in names or ("bwd_dz_gemm" in names and "bwd_grad_gemm" in names)
    assert all(lm.lmhead_profile_record(i)[1] >= 0 for i in range(n))


@pytest.mark.parametrize("tau,wstd", [(0.05, 0.05), (20.0, 0.05), (1.0, 0.4)],
                         ids=["peaked_tau0.05", "flat_tau20", "peaked_weights"])
def test_extreme_temperatures_and_peaked_distributions(tau, wstd):
    """Logits with a wide dynamic range (scaled logits spread over ~100 units,
    so the online maximum moves across tiles and most exponentials underflow)
    and a nearly uniform distribution (entropy close to ln V)."""
    w = _w(520, 256, 3000, 48, tau, "bernoulli", mask_drop=0.2, hidden_dist="rms",
           weight_std=wstd, seed=31)
    x = W.make_inputs(w)
    g = run_gpu(x)
    assert g["fwd_status"] == 0 and g["bwd_status"] == 0
    o = run_oracle(x)
    e = assert_parity(g, o)
    m = x["loss_mask"].numpy() != 0
    if tau == 20.0:
        assert np.all(o["entropy"][m] > np.log(3000) - 0.05)
    else:
        assert np.median(o["entropy"][m]) < 2.0
    print(tau, wstd, e)


def test_soak_back_to_back_steps_bitwise():
    """Forty forward + backward steps back to back on one stream (each kernel
    may start while its predecessor drains and must wait before touching its
    inputs): every step's outputs equal the first step's bit for bit."""
    ensure_built()
    w = _w(1500, 256, 4000, 64, 0.8, "bernoulli", mask_drop=0.3, hidden_dist="rms", seed=61)
    x = W.make_inputs(w)
    g = to_device(x)
    T, H = g["hidden"].shape
    V = g["weight"].shape[0]
    c, tau = x["chunk_size"], x["temperature"]
    ws = torch.empty(max(lm.lmhead_workspace_size(0, T, H, V, c),
                         lm.lmhead_workspace_size(1, T, H, V, c)), dtype=torch.uint8,
                     device="cuda")
    out = {k: torch.empty(T, device="cuda") for k in ("logp", "entropy", "lse")}
    out["d_hidden"] = torch.empty((T, H), device="cuda")
    out["d_weight"] = torch.empty((V, H), device="cuda")
    first = None
    mismatches = []
    for i in range(40):
        rc = lm.lmhead_logps_fwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau, c,
                                 out["logp"], out["entropy"], out["lse"], ws)
        rc |= lm.lmhead_logps_bwd(g["hidden"], g["weight"], g["targets"], g["loss_mask"], tau,
                                  c, g["grad_logp"], g["grad_entropy"], out["lse"],
                                  out["entropy"], out["d_hidden"], out["d_weight"], 0, ws)
        assert rc == 0
        snap = {k: v.clone() for k, v in out.items()}   # stream-ordered copies
        if first is None:
            first = snap
        else:
            for k in out:
                if not torch.equal(snap[k], first[k]):
                    mismatches.append((i, k))
    torch.cuda.synchronize()
    assert lm.lmhead_read_device_status(ws) == 0
    assert not mismatches, mismatches[:10]


def test_forward_token_block_groups():
    """The forward hands out its (token block, vocabulary split) units in
    groups of token blocks; the grouping changes which units run together,
    never a result bit.  A 1 MB budget at H = 512 gives groups of 4 blocks
    of 256 rows over 10 blocks (4, 4, then a ragged 2), which must match the
    plain order bitwise and the oracle within the tolerances."""
    import os
    w = _w(2500, 512, 3000, 64, 0.8, "bernoulli", mask_drop=0.15, hidden_dist="rms",
           weight_std=0.05)
    x = W.make_inputs(w)
    old = os.environ.get("LMHEAD_FWD_GROUP_MB")
    try:
        os.environ["LMHEAD_FWD_GROUP_MB"] = "0"
        plain = run_gpu(x, backward=False)
        os.environ["LMHEAD_FWD_GROUP_MB"] = "1"
        grouped = run_gpu(x, backward=False)
    finally:
        if old is None:
            os.environ.pop("LMHEAD_FWD_GROUP_MB", None)
        else:
            os.environ["LMHEAD_FWD_GROUP_MB"] = old
    for k in ("logp", "entropy", "lse"):
        assert np.array_equal(grouped[k], plain[k]), k
    assert grouped["fwd_status"] == 0
    assert_parity(grouped, run_oracle(x, backward=False), keys=("logp", "entropy", "lse"))


@pytest.mark.parametrize("H", [8192, 16384])
def test_wide_hidden(H):
    """Hidden sizes of large-model heads: long K loops in the forward and dz
    GEMMs, many 256-column output tiles of d_hidden and d_weight, and a token
    block cap (32-40 MB of hidden rows) below the token count.  Two-call
    path and the single call that keeps the logits, against the oracle."""
    from gpu_helpers import run_gpu_fwd_bwd
    w = _w(700, H, 1500, 300, 0.9, "bernoulli", mask_drop=0.2, hidden_dist="rms",
           weight_std=0.01, seed=H)
    x = W.make_inputs(w)
    o = run_oracle(x)
    g = run_gpu(x)
    assert g["fwd_status"] == 0 and g["bwd_status"] == 0
    e = assert_parity(g, o)
    k = run_gpu_fwd_bwd(x, lm.LMHEAD_STRATEGY_KEEP_LOGITS)
    assert k["status"] == 0
    ek = assert_parity(k, o)
    print(H, e, ek)
