"""The single-call forward + backward (lmhead_logps_fwd_bwd): both strategies
against the fp64 oracle, the recompute strategy bit for bit against the two
separate calls, and the keep-logits strategy against the recompute one."""
import numpy as np
import pytest
import torch

from chunked_lm_head_tcgen05_gb300 import workloads as W

from gpu_helpers import assert_parity, rel_fro, run_gpu, run_gpu_fwd_bwd, run_oracle

pytestmark = pytest.mark.gpu

RECOMPUTE, KEEP = 1, 2

CASES = [
    # T, H, V, chunk, tau, mask, extra
    (333, 192, 3001, 300, 0.7, "bernoulli", dict(mask_drop=0.3)),
    (700, 256, 5000, 64, 1.0, "prompt_prefix", dict(rows=2)),
    (257, 320, 1025, 2000, 1.3, "none", {}),
    (1, 128, 100, 1, 1.0, "none", {}),
]


def _x(T, H, V, chunk, tau, mask, extra, seed=5):
    w = W.WORKLOADS["tiny"].with_(T=T, H=H, V=V, chunk_size=chunk, temperature=tau, mask=mask,
                                  seed=seed, hidden_dist="rms", weight_std=0.05, **extra)
    return W.make_inputs(w)


@pytest.mark.parametrize("T,H,V,chunk,tau,mask,extra", CASES,
                         ids=["T%d_H%d_V%d_c%d" % c[:4] for c in CASES])
@pytest.mark.parametrize("strategy", [RECOMPUTE, KEEP], ids=["recompute", "keep_logits"])
def test_against_oracle(T, H, V, chunk, tau, mask, extra, strategy):
    x = _x(T, H, V, chunk, tau, mask, extra)
    g = run_gpu_fwd_bwd(x, strategy)
    assert g["status"] == 0
    assert_parity(g, run_oracle(x))
    if x["loss_mask"] is not None:
        m = x["loss_mask"].numpy() == 0
        for k in ("logp", "entropy", "lse"):
            assert np.all(g[k][m] == 0.0)
        assert np.all(g["d_hidden"][m] == 0.0)


def test_recompute_equals_two_calls_bitwise():
    x = _x(*CASES[0])
    a = run_gpu_fwd_bwd(x, RECOMPUTE)
    b = run_gpu(x)
    for k in ("logp", "entropy", "lse", "d_hidden", "d_weight"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("grad_entropy", [True, False])
def test_keep_logits_matches_recompute(grad_entropy):
    x = _x(1100, 256, 9000, 700, 0.8, "bernoulli", dict(mask_drop=0.15), seed=9)
    a = run_gpu_fwd_bwd(x, RECOMPUTE, grad_entropy=grad_entropy)
    b = run_gpu_fwd_bwd(x, KEEP, grad_entropy=grad_entropy, with_entropy=grad_entropy)
    for k in ("logp", "lse") + (("entropy",) if grad_entropy else ()):
        assert np.abs(a[k] - b[k]).max() < 1e-4, k
    for k in ("d_hidden", "d_weight"):
        assert rel_fro(b[k], a[k]) < 5e-3, k
    o = run_oracle(x, grad_entropy=grad_entropy)
    assert_parity(b, o, keys=("logp", "lse", "d_hidden", "d_weight"))


def test_keep_logits_deterministic_and_accumulates():
    x = _x(520, 128, 2304, 300, 0.9, "packed_pads", dict(pad_tokens=140, segments=5), seed=3)
    a = run_gpu_fwd_bwd(x, KEEP)
    b = run_gpu_fwd_bwd(x, KEEP)
    for k in ("logp", "entropy", "lse", "d_hidden", "d_weight"):
        assert np.array_equal(a[k], b[k]), k
    c = run_gpu_fwd_bwd(x, KEEP, accumulate=True,
                        d_weight_init=torch.from_numpy(a["d_weight"]).float())
    assert rel_fro(c["d_weight"], 2 * a["d_weight"]) < 1e-6


def test_keep_logits_invalid_targets():
    x = _x(150, 64, 600, 600, 1.0, "none", {})
    y = x["targets"].clone()
    y[5], y[77] = 600, -605
    x["targets"] = y
    g = run_gpu_fwd_bwd(x, KEEP)
    assert g["status"] == 6
    assert np.isnan(g["logp"][5]) and np.isnan(g["logp"][77])
    assert_parity(g, run_oracle(x))
