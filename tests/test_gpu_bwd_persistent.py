"""The backward as one persistent launch (tile completion flags between the dz,
dh and dW tiles of all blocks), and as windowed launches (one block's dh and
dW tiles then the next block's dz tiles per launch), against the per-block
path (two launches per block, ordered by the stream), selected with
LMHEAD_BWD_PERSISTENT = 1, 2 and 0.

Both compute every tile from the same operands in the same order, so the
gradients must agree bit for bit; each case is also held to the oracle.
The shapes span several token and vocabulary blocks, a last vocabulary
block narrower than the others, a partial last token block, scattered rows
(masks), accumulation into d_weight, and a step with no scored token."""
import os

import numpy as np
import pytest
import torch

import chunked_lm_head_tcgen05_gb300 as lm
from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import assert_parity, ensure_built, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

TINY = W.WORKLOADS["tiny"]


def _w(T, H, V, chunk, tau, mask="none", seed=11, **kw):
    return TINY.with_(T=T, H=H, V=V, chunk_size=chunk, temperature=tau, mask=mask, seed=seed,
                      hidden_dist="rms", weight_std=0.05, **kw)


def _kernels(fn):
    """Run fn with launch records on; return (result, names of the kernels launched)."""
    ensure_built()
    lm.lmhead_profile_enable(1)
    try:
        out = fn()
        names = {lm.lmhead_profile_record(i)[0] for i in range(lm.lmhead_profile_count())}
    finally:
        lm.lmhead_profile_enable(0)
    return out, names


KERNEL = {"0": "bwd_dz_gemm", "1": "bwd_all_gemm", "2": "bwd_window_gemm"}


def _both(x, **kw):
    """Per-block path, then the persistent launch, then the windowed launches:
    returns (per-block result, persistent result) after checking that the
    windowed result has the persistent result's bits."""
    old = os.environ.get("LMHEAD_BWD_PERSISTENT")
    out = {}
    try:
        for mode in ("0", "1", "2"):
            os.environ["LMHEAD_BWD_PERSISTENT"] = mode
            out[mode], names = _kernels(lambda: run_gpu(x, **kw))
            # each run really took its own path
            assert KERNEL[mode] in names, (mode, names)
            assert not any(KERNEL[m] in names for m in KERNEL if m != mode), (mode, names)
    finally:
        if old is None:
            os.environ.pop("LMHEAD_BWD_PERSISTENT", None)
        else:
            os.environ["LMHEAD_BWD_PERSISTENT"] = old
    _same_bits(out["1"], out["2"])
    return out["0"], out["1"]


def _blocks(x):
    ensure_built()
    T, H = x["hidden"].shape
    V = x["weight"].shape[0]
    _, tb, vb = lm.lmhead_plan_info(T, H, V, x["chunk_size"])
    Ta = (T + 127) // 128 * 128
    return -(-Ta // tb), -(-V // vb), tb, vb


def _same_bits(a, b):
    for k in ("d_hidden", "d_weight"):
        assert a[k].shape == b[k].shape
        diff = np.flatnonzero(a[k].ravel() != b[k].ravel())
        assert diff.size == 0, (k, diff.size, diff[:5])
    assert a["bwd_status"] == 0 and b["bwd_status"] == 0


CASES = [
    # T, H, V, chunk, tau, mask, extra
    (1000, 256, 2800, 64, 0.8, "none", {}),                        # 4 x 6 blocks, narrow last
    (777, 192, 3001, 48, 1.0, "bernoulli", dict(mask_drop=0.35)),  # scattered rows
    (1500, 128, 5000, 40, 0.6, "prompt_prefix", dict(rows=3)),     # many blocks, prefixes
    (300, 320, 1025, 1000, 1.2, "none", {}),                       # one block
]


@pytest.mark.parametrize("T,H,V,chunk,tau,mask,extra", CASES,
                         ids=["T%d_H%d_V%d_c%d" % c[:4] for c in CASES])
def test_persistent_matches_per_block_bitwise(T, H, V, chunk, tau, mask, extra):
    x = W.make_inputs(_w(T, H, V, chunk, tau, mask, **extra))
    a, b = _both(x)
    _same_bits(a, b)
    assert_parity(b, run_oracle(x))
    print(_blocks(x))


def test_several_blocks_and_a_narrow_last_vocabulary_block():
    """The first case really spans token and vocabulary blocks, and its last
    vocabulary block has fewer 256-column tiles than the others."""
    x = W.make_inputs(_w(1000, 256, 2800, 64, 0.8))
    n_tb, n_vb, tb, vb = _blocks(x)
    assert n_tb >= 2 and n_vb >= 3
    V = x["weight"].shape[0]
    last = V - (n_vb - 1) * vb
    assert -(-last // 256) < vb // 256


def test_persistent_accumulate_and_logp_only():
    x = W.make_inputs(_w(900, 128, 2600, 32, 0.9, "bernoulli", mask_drop=0.2))
    V, H = x["weight"].shape
    init = torch.randn((V, H), generator=torch.Generator().manual_seed(5))
    a, b = _both(x, accumulate=True, d_weight_init=init)
    _same_bits(a, b)
    o = run_oracle(x)
    o["d_weight"] = o["d_weight"] + init.double().numpy()
    assert_parity(b, o)
    a, b = _both(x, grad_entropy=False)
    _same_bits(a, b)
    assert_parity(b, run_oracle(x, grad_entropy=False))


def test_persistent_with_no_scored_token():
    """Every row masked: d_hidden and d_weight are exact zeros (d_weight is
    written by the zero-fill of the first token block's dW tiles)."""
    x = W.make_inputs(_w(600, 128, 2000, 32, 1.0))
    x["loss_mask"] = torch.zeros(600, dtype=torch.uint8)
    x["grad_logp"] = torch.zeros(600)
    x["grad_entropy"] = torch.zeros(600)
    V, H = x["weight"].shape
    a, b = _both(x, d_weight_init=torch.full((V, H), 7.0))
    _same_bits(a, b)
    assert np.all(b["d_weight"] == 0.0) and np.all(b["d_hidden"] == 0.0)


def test_persistent_full_size_qwen3_4b_bitwise():
    """The benchmark's workload (T 4096, H 2560, V 151936, chunk 512): the
    two paths agree bit for bit on the whole d_hidden and d_weight."""
    x = W.make_inputs(W.WORKLOADS["qwen3_4b"])
    a, b = _both(x)
    _same_bits(a, b)


def test_more_token_blocks_than_the_flags_hold_fall_back_to_per_block():
    """With 257 token blocks (chunk 1 keeps the blocks at 256 x 256) the
    persistent kernel's flag layout does not apply: the default mode must
    take the per-block path, and the result must still match the oracle."""
    x = W.make_inputs(_w(65792, 64, 512, 1, 0.9, "bernoulli", mask_drop=0.25, seed=21))
    n_tb, n_vb, tb, vb = _blocks(x)
    assert n_tb > 255 and tb == 256
    old = os.environ.pop("LMHEAD_BWD_PERSISTENT", None)
    try:
        g, names = _kernels(lambda: run_gpu(x))
    finally:
        if old is not None:
            os.environ["LMHEAD_BWD_PERSISTENT"] = old
    assert "bwd_dz_gemm" in names and "bwd_all_gemm" not in names, names
    assert g["fwd_status"] == 0 and g["bwd_status"] == 0
    assert_parity(g, run_oracle(x))
